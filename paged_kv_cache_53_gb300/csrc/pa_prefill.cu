// Chunked-prefill attention over paged context on sm_103a tensor cores (tcgen05).
//
// A chunk of prompt tokens attends causally to its sequence's whole context, the chunk
// included ("PagedAttention and Continuous Batching Explained (2026)", section "Chunked
// prefill").  The work is a dense contraction: for KV head h, the (chunk token, query
// head of h's group) pairs form the rows of Q, and each 128-token tile of context is a
// K/V block of the product.
//
// A plan kernel lists one work item per (sequence, KV head, pair of 128-row query
// tiles), heaviest first; CTA i takes item i.  Row r of a query tile is token r / G of
// its slice of the chunk and query head h * G + r % G, so a tile covers 128 / G
// consecutive chunk tokens and every row of it shares the same K/V.  Warp roles:
//   warp 0     TMA producer: both Q tiles once (3-D boxes over [token, head, dim]),
//              then every K/V tile (one 2-D box per block and 64-column half, gathered
//              through the block table, 128-byte swizzle) into a ring of stages.
//   warp 1     MMA issuer (one thread): S_x(j) = Q_x K_j^T into TMEM, then
//              O_x += P_x(j) V_j with P read from TMEM, in the order PV_A(j), S_A(j+1),
//              PV_B(j), S_B(j+1), so that one tile's softmax overlaps the other tile's
//              products.  PV runs in fp16: P rounded to fp16 has a unit roundoff of
//              2^-11, which keeps the output within a 2e-3 absolute bound where bf16's
//              2^-8 would not.  S = Q K^T runs in the input type.  The issuing thread
//              shares its scheduler with two busy softmax warps and gets only part of
//              its issue slots, so it spends as few instructions per MMA as it can
//              (descriptors advanced by constant offsets from precomputed ones).
//   warps 4-11 two softmax warpgroups, one per query tile, one thread per row: read
//              the row of S from TMEM into registers, apply scale and the causal mask,
//              keep the running max (moved only when it grows by more than 2^8,
//              rescaling O in TMEM then) and sum, write P as fp16 over S's own TMEM
//              columns; at the end normalise O and store.
//   warps 2-3, and the softmax warps not on the MMA issuer's scheduler: convert the
//              next step's V tile from bf16 to fp16 in place (exact below 65520 in
//              magnitude; larger values are flagged) and zero the V rows past the
//              context, which would otherwise meet P = 0 with whatever bits they hold.
//              One conversion serves both query tiles.
// Tiles wholly above the diagonal are never loaded.
#include <algorithm>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_launch.h"
#include "pa_tcgen05.cuh"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleThreshold = 8.0f;
constexpr float kNegInf = -__builtin_huge_valf();

struct PrefillItem;

struct PrefillParams {
  void* out;
  PrefillItem* items;  // the work list; the main pass marks items for the exact pass
  int* header;         // [0] items, [1] 1 once any item is marked
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  int32_t* status;
  int max_blocks, num_q_heads, num_kv_heads, group, num_blocks, out_f32;
  float scale_log2;
};

template <int D, int BS, bool PAIR>
struct PrefillCfg {
  // PAIR: a cluster of two CTAs on two SMs shares every product (tcgen05 cta_group::2,
  // M = 256): each CTA holds 128 of the 256 query rows, half of each K tile (64 of its
  // 128 tokens) and half of each V tile (64 of its 128 columns), so that the operand
  // bytes each SM reads from its own shared memory per product, the K/V bytes its TMA
  // writes and the V bytes it converts are all smaller than with one CTA per product.
  static constexpr int kCtas = PAIR ? 2 : 1;
  static constexpr int BM = 128;                       // query rows per tile, per CTA
  static constexpr int kTiles = 2;                     // query tiles per CTA (ping-pong)
  static constexpr int BN = 128;                       // context tokens per K/V tile
  static constexpr int kHalves = D / 64;               // 128-byte column groups of a row
  static constexpr int kQHalfBytes = BM * 128;         // 16 KiB
  static constexpr int kQBytes = kHalves * kQHalfBytes;
  static constexpr int kKRows = BN / kCtas;            // K tile rows (tokens) per CTA
  static constexpr int kKHalfBytes = kKRows * 128;
  static constexpr int kKBytes = kHalves * kKHalfBytes;
  static constexpr int kVHalves = kHalves / kCtas;     // V tile column groups per CTA
  static constexpr int kVHalfBytes = BN * 128;
  static constexpr int kVBytes = kVHalves * kVHalfBytes;
  // separate rings for K and V tiles.  V(j+1) is converted as soon as P(j) is out, and
  // its slot frees only when both P(j-1) V(j-1) products are done: with as many V stages
  // as K stages its load would start about one step before it is needed, less than a
  // load's latency, and the softmax warpgroups would wait for it.  One more V stage starts
  // the load a step earlier.
  static constexpr int kKStages = PAIR ? 3 : (D == 128 ? 2 : 4);
  static constexpr int kVStages = kKStages + 1;
  static constexpr int kBlocksPerTile = BN / BS;
  static constexpr int kKBlocks = kKRows / BS;         // K blocks each CTA loads per tile
  static constexpr int kThreads = 384;                 // producer, MMA, 2 converters, 2 softmax WGs
  static constexpr int kVThreads = 256;                // threads converting V
  static constexpr int kTmemCols = 512;                // S/P_A | S/P_B | O_A | O_B
  // arrivals on the first CTA's v_ready / p_full: one per converting warp / softmax warp
  // of each CTA
  static constexpr int kVReadyArrivals = kVThreads / 32 * kCtas;
  static constexpr int kPFullArrivals = 4 * kCtas;
  // barriers: q_full, k_full[SK], k_empty[SK], v_full[SV], v_empty[SV], v_ready[SV], then
  // per query tile s_full, p_full (first 64 tokens of P), p_full2 (the other 64),
  // pv_done.  K(j) is done with once S(j) has been computed, an iteration before P(j)
  // V(j), so the next K tile loads that much earlier.
  static constexpr int kBars = 1 + 2 * kKStages + 3 * kVStages + 4 * kTiles;
  static constexpr size_t kSmem = 1024 + kTiles * (size_t)kQBytes + kKStages * (size_t)kKBytes +
                                  kVStages * (size_t)kVBytes + kBars * 8 + 16;
};

template <typename T>
struct Fmt;
template <>
struct Fmt<__half> {
  static constexpr int v = 0;
};
template <>
struct Fmt<__nv_bfloat16> {
  static constexpr int v = 1;
};


// ----------------------------------------------------------------------------------
// plan: one work item per (sequence, KV head, pair of query tiles), heaviest first
// ----------------------------------------------------------------------------------
struct PrefillItem {
  int b, h, ctile;
  int wide;  // set by the main pass: a V value of the item is outside fp16's range
};

constexpr int kPlanBuckets = 4096;
constexpr int kPlanThreads = 1024;

// Items are bucketed by how many K/V tiles their later query tile needs (>> key_shift)
// and written in decreasing order, so that CTA i, which takes item i, starts the long
// causal rows first and the grid ends on the short ones.
__global__ void __launch_bounds__(kPlanThreads)
    prefill_plan_kernel(const int32_t* __restrict__ cu_q_lens,
                        const int32_t* __restrict__ context_lens, int num_seqs,
                        int num_kv_heads, int group, int rows_per_item, int bn, int key_shift,
                        long long max_ctx, PrefillItem* __restrict__ items,
                        int* __restrict__ header, int32_t* status) {
  griddep_wait();
  griddep_launch_dependents();
  __shared__ int s_hist[kPlanBuckets];
  __shared__ int s_warp[32];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  for (int i = tid; i < kPlanBuckets; i += blockDim.x) s_hist[i] = 0;
  __syncthreads();
  const int tpt = rows_per_item / group;  // chunk tokens per item
  auto bucket = [&](int ctx0, int chunk, int ct) {
    const int t_last = min(chunk, (ct + 1) * tpt) - 1;
    const int n_kv = (ctx0 + t_last) / bn + 1;
    return kPlanBuckets - 1 - min(kPlanBuckets - 1, n_kv >> key_shift);  // heaviest first
  };
  for (int b = tid; b < num_seqs; b += blockDim.x) {
    const int chunk = cu_q_lens[b + 1] - cu_q_lens[b];
    const int ctx0 = context_lens[b] - chunk;
    if (chunk <= 0) continue;
    if (ctx0 < 0 || context_lens[b] > max_ctx) {  // such a sequence gets no output rows
      flag_status(status, PA_STATUS_BAD_CONTEXT);
      continue;
    }
    const int ncts = (chunk + tpt - 1) / tpt;
    for (int ct = 0; ct < ncts; ++ct) atomicAdd(&s_hist[bucket(ctx0, chunk, ct)], num_kv_heads);
  }
  __syncthreads();
  // exclusive scan of the histogram: each thread owns kPlanBuckets / blockDim buckets
  constexpr int per = kPlanBuckets / kPlanThreads;
  int v[per], run = 0;
#pragma unroll
  for (int k = 0; k < per; ++k) {
    v[k] = s_hist[tid * per + k];
    run += v[k];
  }
  int incl = run;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int t = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += t;
  }
  if (lane == 31) s_warp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    const int w = s_warp[lane];
    int iw = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(~0u, iw, o);
      if (lane >= o) iw += t;
    }
    s_warp[lane] = iw - w;
    if (lane == 31) {
      header[0] = iw;
      header[1] = 0;
    }
  }
  __syncthreads();
  int off = s_warp[wid] + incl - run;
#pragma unroll
  for (int k = 0; k < per; ++k) {
    s_hist[tid * per + k] = off;
    off += v[k];
  }
  __syncthreads();
  for (int b = tid; b < num_seqs; b += blockDim.x) {
    const int chunk = cu_q_lens[b + 1] - cu_q_lens[b];
    const int ctx0 = context_lens[b] - chunk;
    if (chunk <= 0 || ctx0 < 0 || context_lens[b] > max_ctx) continue;
    const int ncts = (chunk + tpt - 1) / tpt;
    for (int ct = 0; ct < ncts; ++ct) {
      const int slot = atomicAdd(&s_hist[bucket(ctx0, chunk, ct)], num_kv_heads);
      for (int h = 0; h < num_kv_heads; ++h) items[slot + h] = PrefillItem{b, h, ct, 0};
    }
  }
}

// Per query tile: where it starts in the chunk and how far it reaches.
struct TileGeom {
  int t0;       // first chunk token
  int ntok;     // chunk tokens in the tile (0: the tile lies past the chunk)
  int n_kv;     // K/V tiles it needs (0 if ntok == 0)
};

// One work item (sequence, KV head, group of query tiles) by one CTA or CTA pair.
// WIDE: the exact pass for items whose V holds values outside fp16's range (bf16 caches
// only): V stays bf16 in shared memory and P enters P V as bf16 hi + lo terms (a relative
// error of 2^-17, as in decode), twice the P V products.
template <typename T, int D, int BS, bool PAIR, bool WIDE>
__device__ __forceinline__ void prefill_item(const CUtensorMap& tmq, const CUtensorMap& tmk,
                                             const CUtensorMap& tmv, const PrefillParams& p,
                                             int it) {
  // a CTA that runs one item (the main pass) gives up the right to allocate tensor memory
  // once it has its columns; the exact pass allocates once per item it takes
  constexpr bool relinquish = !WIDE;
  static_assert(!WIDE || Fmt<T>::v == 1, "the exact pass is for bf16 caches");
  using C = PrefillCfg<D, BS, PAIR>;
  constexpr int BN = C::BN, SK = C::kKStages, SV = C::kVStages, NT = C::kTiles, NC = C::kCtas;
  static_assert(C::kSmem <= 232448, "shared memory per CTA");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base;                              // [tile][half][128 rows][128 B]
  uint8_t* sK = sQ + NT * C::kQBytes;              // [K stage][half][kKRows rows][128 B]
  uint8_t* sV = sK + SK * C::kKBytes;              // [V stage][half][128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + SV * C::kVBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
  // set by a converting thread that met a V value outside fp16's range; read once the
  // item is done
  volatile uint32_t* wide_flag = tmem_slot + 1;
  uint64_t* q_full = bars;
  uint64_t* k_full = bars + 1;
  uint64_t* k_empty = k_full + SK;
  uint64_t* v_full = k_empty + SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* v_ready = v_empty + SV;      // V of the stage converted to fp16
  uint64_t* s_full = v_ready + SV;       // [tile]
  uint64_t* p_full = s_full + NT;        // [tile] P's first half published
  uint64_t* p_full2 = p_full + NT;       // [tile] its second half
  uint64_t* pv_done = p_full2 + NT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int tpt = C::BM / G;  // chunk tokens per query tile of one CTA
  // rank 0 of a pair issues the MMAs; q_full, k_full, p_full and v_ready of rank 0 count
  // both CTAs' copies and arrivals, the other barriers are each CTA's own
  const int crank = PAIR ? (int)cluster_ctarank() : 0;
  const bool leader = crank == 0;
  // waits on barriers the peer CTA may complete take cluster-scope acquire
  auto wait = [](uint64_t* bar, uint32_t parity) {
    return PAIR ? mbar_wait_cluster(smem_addr(bar), parity) : mbar_wait(smem_addr(bar), parity);
  };
  // the address of rank 0's copy of a barrier, for copies and arrivals aimed at it
  auto lead = [](uint64_t* bar) {
    return PAIR ? mapa_shared(smem_addr(bar), 0) : smem_addr(bar);
  };
  // an arrival on rank 0's copy of a barrier
  auto arrive_lead = [&](uint64_t* bar) {
    if (PAIR && !leader) mbar_arrive_remote(lead(bar));
    else mbar_arrive(smem_addr(bar));
  };

  // every exit before the barriers are set up is taken by both CTAs of a pair together
  const PrefillItem item = p.items[it];
  const int h = item.h, b = item.b;
  const int q_begin = __ldg(p.cu_q_lens + b);
  const int chunk = __ldg(p.cu_q_lens + b + 1) - q_begin;
  const int t0_item = item.ctile * NT * NC * tpt;
  if (t0_item >= chunk) return;
  const int ctx = __ldg(p.context_lens + b);
  if (ctx < chunk || (long long)ctx > (long long)p.max_blocks * BS) {
    if (threadIdx.x == 0 && leader && item.ctile == 0 && h == 0)
      flag_status(p.status, PA_STATUS_BAD_CONTEXT);
    return;
  }
  const int ctx0 = ctx - chunk;
  const int nblk_ctx = (ctx + BS - 1) / BS;
  // pg: the product's query tile x (both CTAs' rows), tg: this CTA's rows of it
  TileGeom pg[NT], tg[NT];
#pragma unroll
  for (int x = 0; x < NT; ++x) {
    pg[x].t0 = t0_item + x * NC * tpt;
    pg[x].ntok = max(0, min(NC * tpt, chunk - pg[x].t0));
    pg[x].n_kv = pg[x].ntok > 0 ? (ctx0 + pg[x].t0 + pg[x].ntok - 1) / BN + 1 : 0;
    tg[x].t0 = pg[x].t0 + crank * tpt;
    tg[x].ntok = max(0, min(tpt, chunk - tg[x].t0));
    tg[x].n_kv = pg[x].n_kv;
  }
  const int n_kv = pg[NT - 1].ntok > 0 ? pg[NT - 1].n_kv : pg[0].n_kv;  // the item's K/V tiles

  if (threadIdx.x == 0) {
    *wide_flag = 0;
    mbar_init(smem_addr(q_full), 1);
    for (int i = 0; i < SK; ++i) {
      mbar_init(smem_addr(k_full + i), 1);
      mbar_init(smem_addr(k_empty + i), 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(smem_addr(v_full + i), 1);
      mbar_init(smem_addr(v_empty + i), 1);
      mbar_init(smem_addr(v_ready + i), C::kVReadyArrivals);
    }
    for (int x = 0; x < NT; ++x) {
      mbar_init(smem_addr(s_full + x), 1);
      mbar_init(smem_addr(p_full + x), C::kPFullArrivals);
      mbar_init(smem_addr(p_full2 + x), C::kPFullArrivals);
      mbar_init(smem_addr(pv_done + x), 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      tc::tmem_alloc_pair(smem_addr(tmem_slot), C::kTmemCols);
      if constexpr (relinquish) tc::tmem_relinquish_pair();
    } else {
      tc::tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
      if constexpr (relinquish) tc::tmem_relinquish();
    }
  }
  if (threadIdx.x == 32 + 1) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  tc::fence_before_sync();
  if constexpr (PAIR) cluster_sync();  // both CTAs' barriers exist before either uses them
  else __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S of tile x at x * BN (P_x is written over its first half: token t of
  // the K/V tile in column t / 2, two fp16 per column), O of tile x at NT * BN + x * D.
  bool ok = true;
  // V of K/V tile jv: bf16 -> fp16 in place and rows past the context zeroed, by 256
  // converting threads, each taking every 256th 16-byte piece: warps 2-3 and the six
  // softmax warps that do not share a scheduler (warp index mod 4) with the MMA issuer
  int vt = -1;
  if (warp == 2 || warp == 3) {
    vt = threadIdx.x - 64;
  } else if (warp >= 4 && (warp & 3) != 1) {
    const int q = warp - 4;
    vt = 64 + 32 * (q - (q >= 2 ? 1 : 0) - (q >= 6 ? 1 : 0)) + lane;
  }
  __half2 vmax = __floats2half2_rn(0.f, 0.f);  // largest |v| converted, per lane half
  // called by whole warps
  auto convert_v = [&](int jv) -> bool {
    const int s = jv % SV;
    if (!__all_sync(~0u, mbar_wait(smem_addr(v_full + s), (jv / SV) & 1))) return false;
    const int z0 = ctx - jv * BN;  // rows from z0 on lie past the context
    uint4* sv = reinterpret_cast<uint4*>(sV + s * C::kVBytes);
    constexpr int kPer = C::kVBytes / 16 / C::kVThreads;
    uint4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) v[u] = sv[vt + u * C::kVThreads];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
      // a piece's row: rows are 128 bytes in every 64-column half (the swizzle only
      // permutes pieces within a row); pieces past the context become zeros
      const int i = vt + u * C::kVThreads;
      if (z0 < BN && ((i % (C::kVHalfBytes / 16)) >> 3) >= z0) {
        v[u] = make_uint4(0, 0, 0, 0);
      } else if constexpr (Fmt<T>::v == 1 && !WIDE) {
        uint32_t* w = reinterpret_cast<uint32_t*>(&v[u]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const __half2 hv = __floats2half2_rn(__uint_as_float(w[k] << 16),
                                               __uint_as_float(w[k] & 0xffff0000u));
          vmax = __hmax2(vmax, __habs2(hv));
          w[k] = *reinterpret_cast<const uint32_t*>(&hv);
        }
      }
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) sv[vt + u * C::kVThreads] = v[u];
    tc::fence_proxy_async_smem();  // the tensor core reads what the threads wrote
    __syncwarp();
    if (lane == 0) arrive_lead(v_ready + s);
    return true;
  };

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t keep = l2_policy_evict_last();  // K/V tiles are re-read by other CTAs
    if (lane == 0) {
      int qbytes = 0;
#pragma unroll
      for (int x = 0; x < NT; ++x) qbytes += pg[x].ntok > 0 ? C::kQBytes : 0;
      if (leader) mbar_arrive_expect_tx(smem_addr(q_full), qbytes * NC);
#pragma unroll
      for (int x = 0; x < NT; ++x) {
        if (pg[x].ntok == 0) continue;
#pragma unroll
        for (int hb = 0; hb < C::kHalves; ++hb) {
          const uint32_t dst = smem_addr(sQ + x * C::kQBytes + hb * C::kQHalfBytes);
          if constexpr (PAIR)
            tma_load_3d_pair(dst, &tmq, hb * 64, h * G, q_begin + tg[x].t0, lead(q_full), keep);
          else
            tma_load_3d(dst, &tmq, hb * 64, h * G, q_begin + tg[x].t0, smem_addr(q_full), keep);
        }
      }
    }
    const int32_t* row = p.block_tables + (size_t)b * p.max_blocks;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int bi = j * C::kBlocksPerTile + lane;
      int id = -1;
      if (lane < C::kBlocksPerTile && bi < nblk_ctx) {
        id = __ldg(row + bi);
        if (id < 0 || id >= p.num_blocks) {
          flag_status(p.status, PA_STATUS_BAD_BLOCK);
          id = -1;
        }
      }
      // K of tile j (this CTA's rows of it), once its slot's previous tile is done with
      const int sk = j % SK;
      if (!__all_sync(~0u, wait(k_empty + sk, ((j / SK) & 1) ^ 1))) { ok = false; break; }
      if (lane == 0 && leader) mbar_arrive_expect_tx(smem_addr(k_full + sk), C::kKBytes * NC);
#pragma unroll
      for (int i = 0; i < C::kKBlocks; ++i) {
        const int idi = __shfl_sync(~0u, id, crank * C::kKBlocks + i);
        if (lane == 0) {
          // blocks past the context (and bad ids) read a box wholly outside: zeros
          const int y = idi < 0 ? -BS : (idi * p.num_kv_heads + h) * BS;
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb) {
            const uint32_t dst = smem_addr(sK + sk * C::kKBytes + hb * C::kKHalfBytes + i * BS * 128);
            if constexpr (PAIR) tma_load_2d_pair(dst, &tmk, hb * 64, y, lead(k_full + sk), keep);
            else tma_load_2d(dst, &tmk, hb * 64, y, smem_addr(k_full + sk), keep);
          }
        }
      }
      // V of tile j (this CTA's columns of it) into its own stage
      const int sv = j % SV;
      if (!__all_sync(~0u, wait(v_empty + sv, ((j / SV) & 1) ^ 1))) { ok = false; break; }
      if (lane == 0) mbar_arrive_expect_tx(smem_addr(v_full + sv), C::kVBytes);
#pragma unroll
      for (int i = 0; i < C::kBlocksPerTile; ++i) {
        const int idi = __shfl_sync(~0u, id, i);
        if (lane == 0) {
          const int y = idi < 0 ? -BS : (idi * p.num_kv_heads + h) * BS;
#pragma unroll
          for (int hv = 0; hv < C::kVHalves; ++hv)
            tma_load_2d(smem_addr(sV + sv * C::kVBytes + hv * C::kVHalfBytes + i * BS * 128), &tmv,
                        (crank * C::kVHalves + hv) * 64, y, smem_addr(v_full + sv), keep);
        }
      }
    }
    if (!ok && lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // Order: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), ...  While one tile's softmax runs,
    // the tensor core works through the other tile's P.V and next S.  S_x(j+1) reuses
    // the TMEM columns PV_x(j) reads P from; tcgen05.mma operations issued by one thread
    // execute in order, so no wait is needed between the two.  In a pair only rank 0
    // issues; its commits arrive on the barrier of both CTAs.
    if (leader) {
      // the whole warp runs the loop (waits included, so that it never diverges); one
      // elected lane issues each MMA and commit
      auto wait_w = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(~0u, wait(bar, parity));
      };
      const uint32_t id_s = tc::idesc_f16(Fmt<T>::v, C::BM * NC, BN, false, false);
      // fp16 P and V; bf16 hi + lo P and bf16 V in the exact pass
      const uint32_t id_o = tc::idesc_f16(WIDE ? Fmt<T>::v : Fmt<__half>::v, C::BM * NC, D, false, true);
      auto commit = [](uint64_t* bar) { tc::commit_warp<PAIR>(smem_addr(bar)); };
      // descriptors of each operand's first k-step and first stage, advanced by constant
      // offsets below
      const uint64_t dq0 = tc::smem_desc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(sV), C::kVHalfBytes, 1024);
      auto issue_s = [&](int x, int sk) {
        const uint32_t tS = tmem + x * BN;
        const uint64_t dq = tc::desc_advance(dq0, x * C::kQBytes);
        const uint64_t dk = tc::desc_advance(dk0, sk * C::kKBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          tc::mma_ss_warp<PAIR>(tS, tc::desc_advance(dq, (kk >> 2) * C::kQHalfBytes + koff),
                                tc::desc_advance(dk, (kk >> 2) * C::kKHalfBytes + koff), id_s,
                                kk > 0);
        }
        commit(s_full + x);
      };
      int v_seen = -1;  // last K/V tile whose fp16 V was waited for
      // P_x(j) V(j), in two halves of 64 tokens as the softmax publishes them
      auto issue_pv = [&](int x, int j, int sv, uint32_t vpar) -> bool {
        if (!wait_w(p_full + x, j & 1)) return false;
        if (v_seen < j) {
          if (!wait_w(v_ready + sv, vpar)) return false;
          v_seen = j;
        }
        tc::fence_after_sync();
        const uint32_t tP = tmem + x * BN;
        const uint32_t tO = tmem + NT * BN + x * D;
        const uint64_t dv = tc::desc_advance(dv0, sv * C::kVBytes);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          if (ks == BN / 32) {
            if (!wait_w(p_full2 + x, j & 1)) return false;
            tc::fence_after_sync();
          }
          tc::mma_ts_warp<PAIR>(tO, tP + 8 * ks, tc::desc_advance(dv, ks * 16 * 128), id_o,
                                j > 0 || ks > 0);
          if constexpr (WIDE)  // the lo terms, in columns 64 .. 127
            tc::mma_ts_warp<PAIR>(tO, tP + 64 + 8 * ks, tc::desc_advance(dv, ks * 16 * 128),
                                  id_o, true);
        }
        commit(pv_done + x);
        return true;
      };
      if (!wait_w(q_full, 0) || !wait_w(k_full, 0)) ok = false;
      if (ok) {
        tc::fence_after_sync();
#pragma unroll
        for (int x = 0; x < NT; ++x)
          if (pg[x].n_kv > 0) issue_s(x, 0);
        commit(k_empty);  // K(0) is read once both S(0) are done
      }
      // stages and phase parities of step j's V and step j+1's K, advanced without divisions
      int sv = 0, sk1 = SK > 1 ? 1 : 0;
      uint32_t vpar = 0, kpar1 = SK > 1 ? 0 : 1;
      for (int j = 0; j < n_kv && ok; ++j) {
        bool next_ready = false;
#pragma unroll
        for (int x = 0; x < NT; ++x) {
          if (j < pg[x].n_kv && !issue_pv(x, j, sv, vpar)) { ok = false; break; }
          if (j + 1 < pg[x].n_kv) {
            if (!next_ready) {
              if (!wait_w(k_full + sk1, kpar1)) { ok = false; break; }
              tc::fence_after_sync();
              next_ready = true;
            }
            issue_s(x, sk1);
          }
        }
        commit(v_empty + sv);                          // V(j): both PV(j) issued
        if (j + 1 < n_kv) commit(k_empty + sk1);       // K(j+1): both S
        if (++sv == SV) { sv = 0; vpar ^= 1; }
        if (++sk1 == SK) { sk1 = 0; kpar1 ^= 1; }
      }
      if (!ok && lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp == 2 || warp == 3) {
    for (int jv = 0; jv < n_kv && ok; ++jv)
      if (!convert_v(jv)) ok = false;
    if constexpr (Fmt<T>::v == 1 && !WIDE) {
      // a value at or above 65520 in magnitude became inf (NaN stays NaN): the item is
      // computed again by the exact pass
      const float2 vm = __half22float2(vmax);
      if (!(vm.x < 65504.5f && vm.y < 65504.5f)) {
        *wide_flag = 1;
      }
    }
    if (!ok) flag_status(p.status, PA_STATUS_TIMEOUT);
  } else if (warp >= 4) {
    // --------------------------- softmax / epilogue (one WG per tile) ---------------------------
    const int x = (warp - 4) >> 2;                           // query tile of this warpgroup
    const int r = (threadIdx.x - 128) & 127;                 // row of the tile = TMEM lane
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_bits + x * BN;
    const uint32_t tO = tmem + lane_bits + NT * BN + x * D;
    const TileGeom g = x == 0 ? tg[0] : tg[NT - 1];          // this CTA's rows
    const int rpos = ctx0 + g.t0 + r / G;                    // position of this row's query
    const int rpos_warp = ctx0 + g.t0 + (r & ~31) / G;       // smallest position in the warp
    const float sc = p.scale_log2;
    float m = kNegInf, l = 0.f;
    // V tile 0 before the first step, then tile j+1 after step j
    if (n_kv > 0 && vt >= 0 && !convert_v(0)) ok = false;
    for (int j = 0; j < g.n_kv && ok; ++j) {
      if (!wait(s_full + x, j & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const int kp0 = j * BN;
      const bool full = kp0 + BN - 1 <= rpos_warp;  // below the diagonal for the whole warp
      // the row's scores, loaded behind one wait
      static_assert(BN == 128, "a 128-column row in registers");
      float c[4][32];
#pragma unroll
      for (int k = 0; k < 4; ++k) tc::tmem_ld32(tS + 32 * k, c[k]);
      tc::tmem_wait_ld();
      // row maximum of scale * S over the visible positions
      float mx;
      if (full && sc > 0.f) {
        // four independent chains of three-input maxima: half the instructions of a
        // two-input chain (every instruction of these warps competes for issue slots
        // with the MMA-issuing thread on one of the four schedulers)
        float rm[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          rm[k] = c[k][0];
#pragma unroll
          for (int i = 1; i < 31; i += 2) rm[k] = fmax3f(rm[k], c[k][i], c[k][i + 1]);
          rm[k] = fmaxf(rm[k], c[k][31]);
        }
        mx = fmax3f(rm[0], rm[1], fmaxf(rm[2], rm[3])) * sc;
      } else if (full) {
        mx = kNegInf;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, c[k][i] * sc);
      } else {
        // on the diagonal the scores are scaled in place and masked positions set to -inf
        mx = kNegInf;
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            c[k][i] = kp0 + 32 * k + i <= rpos ? c[k][i] * sc : kNegInf;
            mx = fmaxf(mx, c[k][i]);
          }
      }
      const bool need = mx > m + kRescaleThreshold;
      const float alpha = need ? fast_exp2(m - mx) : 1.f;
      if (need) m = mx;
      // O holds P_0..j-1 V and must be rescaled before P_j V accumulates into it
      const bool rescale = j >= 1 && __any_sync(~0u, need);
      auto publish = [&](uint64_t* bar) {
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) arrive_lead(bar);
      };
      // P = 2^(scale * S - m) in fp16, tokens 32k .. 32k+31 into columns 16k .. 16k+15
      // (the scores there are already in registers).  It is published in two halves of 64
      // tokens (p_full, p_full2) so that the first half's P V products run while the
      // second half is computed; a warp that must rescale O first publishes both halves
      // after it.
      // exponent t = scale * S - m (the diagonal's scores are scaled already: factor 1),
      // two columns per packed FMA (each lane rounds as a scalar fmaf would)
      const float f = full ? sc : 1.f;
      const uint64_t f2x = f2(f, f), negm2 = f2(-m, -m);
      float s2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          float t0, t1;
          f2_split(f2_fma(f2(c[k][2 * i], c[k][2 * i + 1]), f2x, negm2), t0, t1);
          const float e0 = fast_exp2(t0), e1 = fast_exp2(t1);
          s2[i & 3] += e0 + e1;
          if constexpr (WIDE) {
            uint32_t lo;
            pk[i] = Mma<T>::pack_split(e0, e1, lo);
            c[k][i] = __uint_as_float(lo);  // the scores of this chunk are spent
          } else {
            pk[i] = Mma<__half>::pack(e0, e1);
          }
        }
        tc::tmem_st16(tS + 16 * k, pk);
        if constexpr (WIDE) {
          uint32_t lo[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) lo[i] = __float_as_uint(c[k][i]);
          tc::tmem_st16(tS + 64 + 16 * k, lo);
        }
        if ((k & 1) && !rescale) publish(k == 1 ? p_full + x : p_full2 + x);
      }
      l = l * alpha + ((s2[0] + s2[1]) + (s2[2] + s2[3]));
      if (rescale) {
        // once the last of P_0..j-1 V is done
        if (!wait(pv_done + x, (j - 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tc::tmem_ld32(tO + c0, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tc::tmem_st32(tO + c0, o);
        }
        publish(p_full + x);
        publish(p_full2 + x);
      }
      if (j + 1 < n_kv && vt >= 0 && !convert_v(j + 1)) { ok = false; break; }
    }
    // the item's K/V tiles past this tile's last (the other tile reaches further) still
    // need this warpgroup's share of their conversion
    for (int jv = g.n_kv + 1; jv < n_kv && ok && vt >= 0; ++jv)
      if (!convert_v(jv)) ok = false;
    if constexpr (Fmt<T>::v == 1 && !WIDE) {
      // a value at or above 65520 in magnitude became inf (NaN stays NaN): the item is
      // computed again by the exact pass
      const float2 vm = __half22float2(vmax);
      if (!(vm.x < 65504.5f && vm.y < 65504.5f)) {
        *wide_flag = 1;
      }
    }
    // epilogue: O / l -> out rows
    if (ok && g.n_kv > 0 && wait(pv_done + x, (g.n_kv - 1) & 1)) {
      tc::fence_after_sync();
      const float inv = 1.f / l;
      const int rows_valid = g.ntok * G;
      const size_t orow = ((size_t)(q_begin + g.t0 + r / G) * p.num_q_heads + h * G + r % G) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        tc::tmem_ld32(tO + c0, o);
        tc::tmem_wait_ld();
        if (r < rows_valid) {
          if (p.out_f32) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + orow + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv,
                                   o[4 * i + 3] * inv);
          } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<T*>(p.out) + orow + c0);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint32_t w[4];
#pragma unroll
              for (int k = 0; k < 4; ++k)
                w[k] = Mma<T>::pack(o[8 * i + 2 * k] * inv, o[8 * i + 2 * k + 1] * inv);
              dst[i] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          }
        }
      }
    } else if (!ok) {
      flag_status(p.status, PA_STATUS_TIMEOUT);
    }
  }
  griddep_launch_dependents();
  tc::fence_before_sync();
  // in a pair, neither CTA frees its tensor memory or leaves while the other may still
  // write into it or into its barriers
  if constexpr (PAIR) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    if constexpr (PAIR) tc::tmem_dealloc_pair(tmem, C::kTmemCols);
    else tc::tmem_dealloc(tmem, C::kTmemCols);
  }
  if constexpr (Fmt<T>::v == 1 && !WIDE) {
    // the item is computed again by the exact pass (either CTA of a pair may mark it)
    if (threadIdx.x == 0 && *wide_flag != 0) {
      p.items[it].wide = 1;
      p.header[1] = 1;
    }
  }
}

// The main pass: CTA (pair) i takes item i.
template <typename T, int D, int BS, bool PAIR>
__global__ void __launch_bounds__(384, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  griddep_wait();  // the work list and the chunk's K/V (cache write) are complete
  const int it = (int)blockIdx.x / PrefillCfg<D, BS, PAIR>::kCtas;
  if (it >= __ldg(p.header)) return;  // more CTAs launched than items
  prefill_item<T, D, BS, PAIR, false>(tmq, tmk, tmv, p, it);
}

// The exact pass (bf16 caches), launched after the main pass: one wave of CTAs (pairs),
// each looping over the items; all leave at once unless the main pass marked an item.
template <typename T, int D, int BS, bool PAIR>
__global__ void __launch_bounds__(384, 1)
    prefill_wide_kernel(const __grid_constant__ CUtensorMap tmq,
                        const __grid_constant__ CUtensorMap tmk,
                        const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  constexpr int NC = PrefillCfg<D, BS, PAIR>::kCtas;
  griddep_wait();  // the main pass is complete, its marks written
  if (__ldcg(p.header + 1) == 0) {
    griddep_launch_dependents();
    return;
  }
  const int n = __ldcg(p.header);
  for (int it = (int)blockIdx.x / NC; it < n; it += (int)gridDim.x / NC)
    if (__ldcg(&p.items[it].wide) != 0) prefill_item<T, D, BS, PAIR, true>(tmq, tmk, tmv, p, it);
  griddep_launch_dependents();
}

// ----------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------
// Upper bound on the work items of a call: every sequence's chunk at its maximum, in
// items of `rows_per_item` query rows (256 for one CTA, 512 for a pair).
long long prefill_max_items(int num_seqs, int max_q, int num_q_heads, int num_kv_heads,
                            int rows_per_item = 256) {
  const long long per_seq = ((long long)max_q * (num_q_heads / num_kv_heads) + rows_per_item - 1) /
                            rows_per_item;
  return (long long)num_seqs * num_kv_heads * per_seq;
}
constexpr int kMaxDev = 64;
std::mutex g_mutex;

template <typename T, int D, int BS>
int launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  // head dim 128: CTA pairs; head dim 64 (a V half of 32 columns per CTA would not fill
  // a 128-byte swizzle row): one CTA per product
  constexpr bool kPair = D == 128;
  using C = PrefillCfg<D, BS, kPair>;
  static bool configured[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDev)
    return fail(PA_ERR_CUDA, "pa_prefill_chunk: no usable device");
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!configured[dev]) {
      bool ok = cudaFuncSetAttribute(prefill_kernel<T, D, BS, kPair>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)C::kSmem) == cudaSuccess;
      if constexpr (Fmt<T>::v == 1)
        ok = ok && cudaFuncSetAttribute(prefill_wide_kernel<T, D, BS, kPair>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)C::kSmem) == cudaSuccess;
      if (!ok) return fail(PA_ERR_CUDA, "pa_prefill_chunk: shared-memory configuration failed");
      configured[dev] = true;
    }
  }
  const int G = a.num_q_heads / a.num_kv_heads;
  CUtensorMap tmq, tmk, tmv;
  const int r0 = encode_query_map(&tmq, a.q, a.dtype, a.num_tokens, a.num_q_heads, a.head_dim, G,
                                  C::BM / G);
  const int r1 = encode_cache_map(&tmk, a.k_cache, a.dtype, a.num_blocks, a.num_kv_heads,
                                  a.block_size, a.head_dim);
  const int r2 = encode_cache_map(&tmv, a.v_cache, a.dtype, a.num_blocks, a.num_kv_heads,
                                  a.block_size, a.head_dim);
  if (r0 != CUDA_SUCCESS || r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS)
    return fail(PA_ERR_CUDA, "pa_prefill_chunk: cuTensorMapEncodeTiled failed (%d, %d, %d)", r0,
                r1, r2);
  PrefillParams p;
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.cu_q_lens = a.cu_q_lens;
  p.context_lens = a.context_lens;
  p.status = a.status;
  p.max_blocks = a.max_blocks;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = G;
  p.num_blocks = a.num_blocks;
  p.out_f32 = a.out_dtype == PA_F32;
  p.scale_log2 = a.scale * kLog2e;
  const int rows_per_item = C::BM * C::kTiles * C::kCtas;
  const long long items = prefill_max_items(a.num_seqs, a.max_q, a.num_q_heads, a.num_kv_heads,
                                            rows_per_item);
  if (items * C::kCtas > 0x7fffffffll)
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill_chunk: grid too large");
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.header = reinterpret_cast<int*>(ws);
  p.items = reinterpret_cast<PrefillItem*>(ws + 256);
  int key_shift = 0;
  while (((long long)a.max_ctx / C::BN + 1) >> key_shift >= kPlanBuckets) ++key_shift;
  cudaError_t e = launch_pdl(prefill_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream,
                             a.cu_q_lens, a.context_lens, a.num_seqs, a.num_kv_heads, G,
                             rows_per_item, C::BN, key_shift,
                             std::min<long long>(a.max_ctx, (long long)a.max_blocks * a.block_size),
                             reinterpret_cast<PrefillItem*>(ws + 256), reinterpret_cast<int*>(ws),
                             a.status);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_prefill_chunk (plan): %s", cudaGetErrorString(e));
  e = launch_pdl_cluster(prefill_kernel<T, D, BS, kPair>, dim3((unsigned)(items * C::kCtas)),
                         dim3(C::kThreads), C::kSmem, stream, C::kCtas, tmq, tmk, tmv, p);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_prefill_chunk: %s", cudaGetErrorString(e));
  if constexpr (Fmt<T>::v == 1) {
    // bf16: the exact pass for items whose V does not fit fp16 (one wave, idle otherwise)
    const long long wave = std::max(1, sm_count() / C::kCtas);
    const long long n = std::min<long long>(items, wave) * C::kCtas;
    e = launch_pdl_cluster(prefill_wide_kernel<T, D, BS, kPair>, dim3((unsigned)n),
                           dim3(C::kThreads), C::kSmem, stream, C::kCtas, tmq, tmk, tmv, p);
    if (e != cudaSuccess)
      return fail(PA_ERR_CUDA, "pa_prefill_chunk (exact pass): %s", cudaGetErrorString(e));
  }
  return PA_OK;
}

template <typename T>
int dispatch(const PrefillArgs& a, cudaStream_t stream) {
  if (a.head_dim == 128 && a.block_size == 16) return launch_prefill_t<T, 128, 16>(a, stream);
  if (a.head_dim == 128 && a.block_size == 32) return launch_prefill_t<T, 128, 32>(a, stream);
  if (a.head_dim == 64 && a.block_size == 16) return launch_prefill_t<T, 64, 16>(a, stream);
  if (a.head_dim == 64 && a.block_size == 32) return launch_prefill_t<T, 64, 32>(a, stream);
  return fail(PA_ERR_UNSUPPORTED, "pa_prefill_chunk: head_dim %d / block_size %d", a.head_dim,
              a.block_size);
}

}  // namespace

size_t prefill_workspace_bytes(int num_seqs, int, int max_q, int num_q_heads, int num_kv_heads,
                               int, int, int) {
  return 256 + sizeof(PrefillItem) *
                   (size_t)prefill_max_items(num_seqs, max_q, num_q_heads, num_kv_heads);
}

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? dispatch<__nv_bfloat16>(a, stream) : dispatch<__half>(a, stream);
}

}  // namespace pa
