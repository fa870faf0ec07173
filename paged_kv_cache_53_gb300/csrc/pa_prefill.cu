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
//              products.  P is carried as the sum of a bf16/fp16 "hi" term and its
//              rounding residual "lo" (two MMAs): a single 16-bit P alone can miss a 2e-3
//              absolute tolerance on short contexts.
//   warps 4-11 two softmax warpgroups, one per query tile, one thread per row: read
//              S from TMEM, apply scale and the causal mask, keep the running max
//              (moved only when it grows by more than 2^8, rescaling O in TMEM then) and
//              sum, write P over S's own TMEM columns; at the end normalise O and store.
// Tiles wholly above the diagonal are never loaded; only the last K/V tile can hold
// positions past the context, whose V rows are zeroed before they meet P = 0.
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
  const PrefillItem* items;
  const int* header;
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  int32_t* status;
  int max_blocks, num_q_heads, num_kv_heads, group, num_blocks, out_f32;
  float scale_log2;
};

template <int D, int BS>
struct PrefillCfg {
  static constexpr int BM = 128;                       // query rows per tile
  static constexpr int kTiles = 2;                     // query tiles per CTA (ping-pong)
  static constexpr int BN = 128;                       // context tokens per K/V tile
  static constexpr int kHalves = D / 64;               // 128-byte column groups
  static constexpr int kQHalfBytes = BM * 128;         // 16 KiB
  static constexpr int kQBytes = kHalves * kQHalfBytes;
  static constexpr int kKvHalfBytes = BN * 128;        // 16 KiB
  static constexpr int kKBytes = kHalves * kKvHalfBytes;
  static constexpr int kStageBytes = 2 * kKBytes;      // K then V
  static constexpr int kStages = D == 128 ? 2 : 4;
  static constexpr int kBlocksPerTile = BN / BS;
  static constexpr int kThreads = 384;                 // producer, MMA, 2 idle, 2 x softmax WG
  static constexpr int kTmemCols = 512;                // S/P_A | S/P_B | O_A | O_B
  // barriers: q_full, kv_full[S], kv_empty[S], then per query tile s_full, p_full, pv_done
  static constexpr int kBars = 1 + 2 * kStages + 3 * kTiles;
  static constexpr size_t kSmem = 1024 + kTiles * (size_t)kQBytes + (size_t)kStages * kStageBytes +
                                  kBars * 8 + 16;
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

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ----------------------------------------------------------------------------------
// plan: one work item per (sequence, KV head, pair of query tiles), heaviest first
// ----------------------------------------------------------------------------------
struct PrefillItem {
  int b, h, ctile, pad;
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
    if (lane == 31) header[0] = iw;
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

// Per query tile of a CTA: where it starts in the chunk and how far it reaches.
struct TileGeom {
  int t0;       // first chunk token
  int ntok;     // chunk tokens in the tile (0: the tile lies past the chunk)
  int n_kv;     // K/V tiles it needs (0 if ntok == 0)
};

template <typename T, int D, int BS>
__global__ void __launch_bounds__(384, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  using C = PrefillCfg<D, BS>;
  constexpr int BN = C::BN, S = C::kStages, NT = C::kTiles;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base;                              // [tile][half][128 rows][128 B]
  uint8_t* sKV = sQ + NT * C::kQBytes;             // [stage][K | V][half][128 rows][128 B]
  uint64_t* bars = reinterpret_cast<uint64_t*>(sKV + S * C::kStageBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + S;
  uint64_t* s_full = bars + 1 + 2 * S;  // [tile]
  uint64_t* p_full = s_full + NT;
  uint64_t* pv_done = p_full + NT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.group;
  const int tpt = C::BM / G;  // chunk tokens per query tile

  griddep_wait();  // the work list and the chunk's K/V (cache write) are complete
  if ((int)blockIdx.x >= __ldg(p.header)) return;  // more CTAs launched than items
  const PrefillItem item = p.items[blockIdx.x];
  const int h = item.h, b = item.b;
  const int q_begin = __ldg(p.cu_q_lens + b);
  const int chunk = __ldg(p.cu_q_lens + b + 1) - q_begin;
  const int t0_cta = item.ctile * NT * tpt;
  if (t0_cta >= chunk) return;  // the whole CTA leaves before touching any barrier
  const int ctx = __ldg(p.context_lens + b);
  if (ctx < chunk || (long long)ctx > (long long)p.max_blocks * BS) {
    if (threadIdx.x == 0 && item.ctile == 0 && h == 0) flag_status(p.status, PA_STATUS_BAD_CONTEXT);
    return;
  }
  const int ctx0 = ctx - chunk;
  const int nblk_ctx = (ctx + BS - 1) / BS;
  TileGeom tg[NT];
#pragma unroll
  for (int x = 0; x < NT; ++x) {
    tg[x].t0 = t0_cta + x * tpt;
    tg[x].ntok = max(0, min(tpt, chunk - tg[x].t0));
    tg[x].n_kv = tg[x].ntok > 0 ? (ctx0 + tg[x].t0 + tg[x].ntok - 1) / BN + 1 : 0;
  }
  const int n_kv = tg[NT - 1].ntok > 0 ? tg[NT - 1].n_kv : tg[0].n_kv;  // the CTA's K/V tiles

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(q_full), 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_addr(kv_full + i), 1);
      mbar_init(smem_addr(kv_empty + i), 1);
    }
    for (int x = 0; x < NT; ++x) {
      mbar_init(smem_addr(s_full + x), 1);
      mbar_init(smem_addr(p_full + x), 128);
      mbar_init(smem_addr(pv_done + x), 1);
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 32 + 1) {
    prefetch_tensormap(&tmq);
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  // TMEM columns: S of tile x at x * BN (P_x is written over it), O of tile x at
  // NT * BN + x * D.  P layout: 32-token chunk c of the row holds its 16-bit hi terms in
  // columns 32c .. 32c+15 and its lo terms in 32c+16 .. 32c+31 (two tokens per column).
  bool ok = true;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t keep = l2_policy_evict_last();  // K/V tiles are re-read by other CTAs
    if (lane == 0) {
      int qbytes = 0;
#pragma unroll
      for (int x = 0; x < NT; ++x) qbytes += tg[x].ntok > 0 ? C::kQBytes : 0;
      mbar_arrive_expect_tx(smem_addr(q_full), qbytes);
#pragma unroll
      for (int x = 0; x < NT; ++x) {
        if (tg[x].ntok == 0) continue;
#pragma unroll
        for (int hb = 0; hb < C::kHalves; ++hb)
          tma_load_3d(smem_addr(sQ + x * C::kQBytes + hb * C::kQHalfBytes), &tmq, hb * 64, h * G,
                      q_begin + tg[x].t0, smem_addr(q_full), keep);
      }
    }
    const int32_t* row = p.block_tables + (size_t)b * p.max_blocks;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int s = j % S;
      if (!mbar_wait(smem_addr(kv_empty + s), ((j / S) & 1) ^ 1)) { ok = false; break; }
      const int bi = j * C::kBlocksPerTile + lane;
      int id = -1;
      if (lane < C::kBlocksPerTile && bi < nblk_ctx) {
        id = __ldg(row + bi);
        if (id < 0 || id >= p.num_blocks) {
          flag_status(p.status, PA_STATUS_BAD_BLOCK);
          id = -1;
        }
      }
      uint8_t* st = sKV + s * C::kStageBytes;
      if (lane == 0) mbar_arrive_expect_tx(smem_addr(kv_full + s), C::kStageBytes);
#pragma unroll
      for (int i = 0; i < C::kBlocksPerTile; ++i) {
        const int idi = __shfl_sync(~0u, id, i);
        if (lane == 0) {
          // blocks past the context (and bad ids) read a box wholly outside: zeros
          const int y = idi < 0 ? -BS : (idi * p.num_kv_heads + h) * BS;
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb) {
            const int off = hb * C::kKvHalfBytes + i * BS * 128;
            tma_load_2d(smem_addr(st + off), &tmk, hb * 64, y, smem_addr(kv_full + s), keep);
            tma_load_2d(smem_addr(st + C::kKBytes + off), &tmv, hb * 64, y,
                        smem_addr(kv_full + s), keep);
          }
        }
      }
    }
    if (!ok && lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // Order: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), ...  While one tile's softmax runs,
    // the tensor core works through the other tile's P.V and next S.  S_x(j+1) reuses
    // the TMEM columns PV_x(j) reads P from; tcgen05.mma operations issued by one thread
    // execute in order, so no wait is needed between the two.
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_f16(Fmt<T>::v, C::BM, BN, false, false);
      const uint32_t id_o = tc::idesc_f16(Fmt<T>::v, C::BM, D, false, true);
      auto issue_s = [&](int x, int j) {
        const uint32_t tS = tmem + x * BN;
        const uint32_t sq = smem_addr(sQ + x * C::kQBytes);
        const uint32_t sk = smem_addr(sKV + (j % S) * C::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          const uint64_t a = tc::smem_desc_sw128(sq + (kk >> 2) * C::kQHalfBytes + koff, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(sk + (kk >> 2) * C::kKvHalfBytes + koff, 16, 1024);
          tc::mma_f16_ss(tS, a, bd, id_s, kk > 0);
        }
        tc::commit(smem_addr(s_full + x));
      };
      auto issue_pv = [&](int x, int j) -> bool {
        if (!mbar_wait(smem_addr(p_full + x), j & 1)) return false;
        tc::fence_after_sync();
        const uint32_t tP = tmem + x * BN;
        const uint32_t tO = tmem + NT * BN + x * D;
        const uint32_t sv = smem_addr(sKV + (j % S) * C::kStageBytes + C::kKBytes);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint32_t col = 32 * (ks >> 1) + 8 * (ks & 1);
          const uint64_t bdesc = tc::smem_desc_sw128(sv + ks * 16 * 128, C::kKvHalfBytes, 1024);
          tc::mma_f16_ts(tO, tP + col, bdesc, id_o, j > 0 || ks > 0);
          tc::mma_f16_ts(tO, tP + col + 16, bdesc, id_o, true);
        }
        tc::commit(smem_addr(pv_done + x));
        return true;
      };
      if (!mbar_wait(smem_addr(q_full), 0) || !mbar_wait(smem_addr(kv_full), 0)) ok = false;
      if (ok) {
        tc::fence_after_sync();
#pragma unroll
        for (int x = 0; x < NT; ++x)
          if (tg[x].n_kv > 0) issue_s(x, 0);
      }
      for (int j = 0; j < n_kv && ok; ++j) {
        bool next_ready = false;
#pragma unroll
        for (int x = 0; x < NT; ++x) {
          if (j < tg[x].n_kv && !issue_pv(x, j)) { ok = false; break; }
          if (j + 1 < tg[x].n_kv) {
            if (!next_ready) {
              if (!mbar_wait(smem_addr(kv_full + (j + 1) % S), ((j + 1) / S) & 1)) { ok = false; break; }
              tc::fence_after_sync();
              next_ready = true;
            }
            issue_s(x, j + 1);
          }
        }
        tc::commit(smem_addr(kv_empty + j % S));
      }
      if (!ok) flag_status(p.status, PA_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // --------------------------- softmax / epilogue (one WG per tile) ---------------------------
    const int x = (warp - 4) >> 2;                           // query tile of this warpgroup
    const int r = (threadIdx.x - 128) & 127;                 // row of the tile = TMEM lane
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_bits + x * BN;
    const uint32_t tO = tmem + lane_bits + NT * BN + x * D;
    const TileGeom g = x == 0 ? tg[0] : tg[NT - 1];
    const int rpos = ctx0 + g.t0 + r / G;                    // position of this row's query
    const int rpos_warp = ctx0 + g.t0 + (r & ~31) / G;       // smallest position in the warp
    const float sc = p.scale_log2;
    float m = kNegInf, l = 0.f;
    for (int j = 0; j < g.n_kv; ++j) {
      if (!mbar_wait(smem_addr(s_full + x), j & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const int kp0 = j * BN;
      const bool full = kp0 + BN - 1 <= rpos_warp;  // below the diagonal for the whole warp
      // pass 1: row maximum of scale * S over the visible positions
      float mx = kNegInf;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 64) {
        float a[32], bq[32];
        tc::tmem_ld32(tS + c0, a);
        tc::tmem_ld32(tS + c0 + 32, bq);
        tc::tmem_wait_ld();
        if (full) {
#pragma unroll
          for (int i = 0; i < 32; ++i) mx = fmaxf(mx, fmaxf(a[i], bq[i]) * sc);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            mx = fmaxf(mx, kp0 + c0 + i <= rpos ? a[i] * sc : kNegInf);
            mx = fmaxf(mx, kp0 + c0 + 32 + i <= rpos ? bq[i] * sc : kNegInf);
          }
        }
      }
      const bool need = mx > m + kRescaleThreshold;
      const float alpha = need ? fast_exp2(m - mx) : 1.f;
      if (need) m = mx;
      // pass 2: P = 2^(scale * S - m) as hi + lo 16-bit terms, over S's own columns
      float sum = 0.f;
#pragma unroll
      for (int c0 = 0; c0 < BN; c0 += 32) {
        float a[32];
        tc::tmem_ld32(tS + c0, a);
        tc::tmem_wait_ld();
        if (full) {
#pragma unroll
          for (int i = 0; i < 32; ++i) a[i] = fast_exp2(fmaf(a[i], sc, -m));
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            a[i] = kp0 + c0 + i <= rpos ? fast_exp2(fmaf(a[i], sc, -m)) : 0.f;
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          sum += a[2 * i] + a[2 * i + 1];
          hi[i] = Mma<T>::pack_split(a[2 * i], a[2 * i + 1], lo[i]);
        }
        tc::tmem_st16(tS + c0, hi);
        tc::tmem_st16(tS + c0 + 16, lo);
      }
      l = l * alpha + sum;
      if (j >= 1 && __any_sync(~0u, need)) {
        // O holds P_0..j-1 V: once the last of those products is done, rescale it
        if (!mbar_wait(smem_addr(pv_done + x), (j - 1) & 1)) { ok = false; break; }
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
      }
      // V rows of the context's last K/V tile past the context (inside its last block)
      // may hold anything, NaN bits included, and would meet P = 0: zero them.  Both
      // warpgroups may do it; they write the same zeros.
      const int z0 = ctx - kp0, z1 = min(BN, nblk_ctx * BS - kp0);
      if (z0 < z1) {
        const int s = j % S;
        if (!mbar_wait(smem_addr(kv_full + s), (j / S) & 1)) { ok = false; break; }
        const uint32_t sv = smem_addr(sKV + s * C::kStageBytes + C::kKBytes);
        for (int i = r; i < (z1 - z0) * (D / 8); i += 128) {
          const int vr = z0 + i / (D / 8), c = i % (D / 8);
          st_shared_v4(sv + (c >> 3) * C::kKvHalfBytes + vr * 128 + (c & 7) * 16,
                       make_uint4(0, 0, 0, 0));
        }
        tc::fence_proxy_async_smem();
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(smem_addr(p_full + x));
    }
    // epilogue: O / l -> out rows
    if (ok && g.n_kv > 0 && mbar_wait(smem_addr(pv_done + x), (g.n_kv - 1) & 1)) {
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
  __syncthreads();
  if (warp == 1) {
    tc::fence_after_sync();
    tc::tmem_dealloc(tmem, C::kTmemCols);
  }
}

// ----------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------
// Upper bound on the work items of a call: every sequence's chunk at its maximum.
long long prefill_max_items(int num_seqs, int max_q, int num_q_heads, int num_kv_heads) {
  const long long rows_per_item = 128 * 2;  // PrefillCfg<>::BM * kTiles
  const long long per_seq = ((long long)max_q * (num_q_heads / num_kv_heads) + rows_per_item - 1) /
                            rows_per_item;
  return (long long)num_seqs * num_kv_heads * per_seq;
}
constexpr int kMaxDev = 64;
std::mutex g_mutex;

template <typename T, int D, int BS>
int launch_prefill_t(const PrefillArgs& a, cudaStream_t stream) {
  using C = PrefillCfg<D, BS>;
  static bool configured[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDev)
    return fail(PA_ERR_CUDA, "pa_prefill_chunk: no usable device");
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(prefill_kernel<T, D, BS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)C::kSmem) != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_prefill_chunk: shared-memory configuration failed");
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
  const long long items = prefill_max_items(a.num_seqs, a.max_q, a.num_q_heads, a.num_kv_heads);
  if (items > 0x7fffffffll) return fail(PA_ERR_UNSUPPORTED, "pa_prefill_chunk: grid too large");
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.header = reinterpret_cast<int*>(ws);
  p.items = reinterpret_cast<const PrefillItem*>(ws + 256);
  int key_shift = 0;
  while (((long long)a.max_ctx / C::BN + 1) >> key_shift >= kPlanBuckets) ++key_shift;
  cudaError_t e = launch_pdl(prefill_plan_kernel, dim3(1), dim3(kPlanThreads), 0, stream,
                             a.cu_q_lens, a.context_lens, a.num_seqs, a.num_kv_heads, G,
                             C::BM * C::kTiles, C::BN, key_shift,
                             std::min<long long>(a.max_ctx, (long long)a.max_blocks * a.block_size),
                             reinterpret_cast<PrefillItem*>(ws + 256), reinterpret_cast<int*>(ws),
                             a.status);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_prefill_chunk (plan): %s", cudaGetErrorString(e));
  e = launch_pdl(prefill_kernel<T, D, BS>, dim3((unsigned)items), dim3(C::kThreads), C::kSmem,
                 stream, tmq, tmk, tmv, p);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_prefill_chunk: %s", cudaGetErrorString(e));
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
