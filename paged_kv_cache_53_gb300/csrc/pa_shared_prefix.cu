// Attention of one shared prefix for every sequence that reads it, on sm_103a tensor
// cores (tcgen05).
//
// When many sequences point their tables at the same physical prefix blocks ("Continuous
// batching, paged attention, prefix caching", section "Prefix caching"), their decode
// queries all attend to the same prefix K/V.  Per KV head h, the query groups of all the
// sharers form the rows of one dense product with the prefix's K/V, so the prefix is read
// once instead of once per sequence.  This kernel computes, for each sharer and each
// piece ("split") of the prefix, the partial (running max, sum, unnormalised output) in
// the same form as the decode kernels' split-KV partials, into slots the decode plan
// reserved ahead of the sharer's own partitions; the decode merge then combines them.
//
// CTA (pair, split, h) owns two 128-row query tiles; row r of the pair is sharer
// (pair * 256 + r) / G, query head h * G + r % G.  The pipeline is the chunked-prefill
// kernel's: a TMA producer warp streams 128-token K and V tiles of the prefix through the
// prefix's block list into a K ring and a V ring; one warp issues S = Q K^T and O += P V with P written
// into S's TMEM columns; two softmax warpgroups, one per query tile, run the online
// softmax.  The query rows are gathered from scattered sequences, so every thread of the
// CTA copies a share of them into 128-byte-swizzled shared memory before the pipeline
// starts.  No causal mask: every row sees the whole split.
// P V: for fp16 caches P is one fp16 term (unit roundoff 2^-11) against V as stored; for
// bf16 caches P is a pair of bf16 hi + lo terms (a relative error of 2^-17, twice the
// products) against V as stored, bf16 having too few bits for P alone.  (Converting each
// bf16 V tile to fp16 in place, by two warps, so that one fp16 P term would do, made
// every step longer than the halved products saved.)
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

template <int D, int BS>
struct SpCfg {
  static constexpr int BM = 128, kTiles = 2, BN = 128;
  static constexpr int kHalves = D / 64;
  static constexpr int kQHalfBytes = BM * 128;
  static constexpr int kQBytes = kHalves * kQHalfBytes;
  static constexpr int kKvHalfBytes = BN * 128;
  static constexpr int kKBytes = kHalves * kKvHalfBytes;  // one K (or V) tile
  // K and V tiles in rings of their own: K(j) is free once both S(j) products are done,
  // a step before V(j), so its next tile loads a step earlier than in a shared ring
  static constexpr int kKStages = D == 128 ? 2 : 4;
  static constexpr int kVStages = D == 128 ? 2 : 4;
  static constexpr int kBlocksPerTile = BN / BS;
  static constexpr int kThreads = 384;
  static constexpr int kTmemCols = 512;
  // k_full[SK], k_empty[SK], v_full[SV], v_empty[SV], then per query tile s_full, p_full,
  // pv_done, then q_full
  static constexpr int kBars = 2 * kKStages + 2 * kVStages + 3 * kTiles + 1;
  static constexpr int kGatherThreads = kThreads - 32;  // every warp but the producer
  static constexpr int kMaxSharers = kTiles * BM;  // sequences whose rows one CTA takes
  static constexpr size_t kSmem = 1024 + kTiles * (size_t)kQBytes +
                                  (size_t)(kKStages + kVStages) * kKBytes + kBars * 8 + 16 +
                                  kMaxSharers * 4;
};

template <typename T>
struct SpFmt;
template <>
struct SpFmt<__half> {
  static constexpr int v = 0;
};
template <>
struct SpFmt<__nv_bfloat16> {
  static constexpr int v = 1;
};

struct SpParams {
  const void* q;
  const int32_t* sharers;
  const int32_t* prefix_blocks;
  const int* part_start;
  float2* part_ml;
  float* part_acc;
  int32_t* status;
  int num_sharers, prefix_len, split_tokens;
  int num_seqs, num_q_heads, num_kv_heads, group, num_blocks;
  float scale_log2;
};

template <typename T, int D, int BS>
__global__ void __launch_bounds__(384, 1)
    shared_prefix_kernel(const __grid_constant__ CUtensorMap tmk,
                         const __grid_constant__ CUtensorMap tmv, const SpParams p) {
  using C = SpCfg<D, BS>;
  constexpr int BN = C::BN, SK = C::kKStages, SV = C::kVStages, NT = C::kTiles;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sK = sQ + NT * C::kQBytes;
  uint8_t* sV = sK + SK * C::kKBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sV + SV * C::kKBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
  int* s_seq = reinterpret_cast<int*>(tmem_slot + 4);  // [kMaxSharers]
  uint64_t* k_full = bars;
  uint64_t* k_empty = bars + SK;
  uint64_t* v_full = bars + 2 * SK;
  uint64_t* v_empty = v_full + SV;
  uint64_t* s_full = v_empty + SV;
  uint64_t* p_full = s_full + NT;
  uint64_t* pv_done = p_full + NT;
  uint64_t* q_full = pv_done + NT;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = blockIdx.x, split = blockIdx.y, h = blockIdx.z;
  const int G = p.group;
  const int rows_total = p.num_sharers * G;
  const int row0 = pair * NT * C::BM;
  const int kv_begin = split * p.split_tokens;
  const int kv_end = min(p.prefix_len, kv_begin + p.split_tokens);
  const int n_kv = (kv_end - kv_begin + BN - 1) / BN;
  const int nblk = p.prefix_len / BS;

  // the sequences of this CTA's sharers (G query rows each), read while the barriers and the
  // tensor memory are set up: -1 for an index out of range (the decode plan flags it)
  const int si_lo = row0 / G;
  const int si_hi = min(p.num_sharers, (row0 + NT * C::BM + G - 1) / G);
  for (int i = threadIdx.x; si_lo + i < si_hi; i += C::kThreads) {
    const int sb = __ldg(p.sharers + si_lo + i);
    s_seq[i] = sb >= 0 && sb < p.num_seqs ? sb : -1;
  }
  if (threadIdx.x == 0) {
    for (int i = 0; i < SK; ++i) {
      mbar_init(smem_addr(k_full + i), 1);
      mbar_init(smem_addr(k_empty + i), 1);
    }
    for (int i = 0; i < SV; ++i) {
      mbar_init(smem_addr(v_full + i), 1);
      mbar_init(smem_addr(v_empty + i), 1);
    }
    for (int x = 0; x < NT; ++x) {
      mbar_init(smem_addr(s_full + x), 1);
      mbar_init(smem_addr(p_full + x), 128);
      mbar_init(smem_addr(pv_done + x), 1);
    }
    mbar_init(smem_addr(q_full), C::kGatherThreads);
    fence_mbar_init();
  }
  if (warp == 1) {
    tc::tmem_alloc(smem_addr(tmem_slot), C::kTmemCols);
    tc::tmem_relinquish();
  }
  if (threadIdx.x == 33) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  // the attention kernel, launched next, waits for the plan through a flag of its own and
  // for this grid only on its way out: it may start now, on the SMs this grid leaves free
  griddep_launch_dependents();
  const uint32_t tmem = *tmem_slot;
  bool valid[NT];
#pragma unroll
  for (int x = 0; x < NT; ++x) valid[x] = row0 + x * C::BM < rows_total;
  bool ok = true;
  // Only the partial slots (part_start) come from the decode plan, the kernel launched just
  // before this one; the epilogue waits for it.  The query rows and the prefix's K/V were
  // written before the plan started (it waits for its own predecessors before letting
  // this kernel launch), so they are read while the plan still runs.

  if (warp > 0) {
    // the query rows of both tiles, gathered from their sequences into the 128-byte
    // swizzled layout while the producer's first K/V tiles are in flight (rows past the
    // sharers read zeros); every load of a thread in flight at once
    constexpr int kItems = NT * C::BM * (D / 8);
    constexpr int kUnroll = (kItems + C::kGatherThreads - 1) / C::kGatherThreads;
    const int t = threadIdx.x - 32;
    for (int i0 = t; i0 < kItems; i0 += kUnroll * C::kGatherThreads) {
      uint4 v[kUnroll];
      uint32_t off[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int idx = i0 + u * C::kGatherThreads;
        const int rr = idx / (D / 8), c = idx - rr * (D / 8);
        const int x = rr / C::BM, r = rr - x * C::BM;
        const int grow = row0 + rr;
        v[u] = make_uint4(0, 0, 0, 0);
        off[u] = idx < kItems ? (uint32_t)(x * C::kQBytes + (c >> 3) * C::kQHalfBytes + r * 128 +
                                           (((c & 7) ^ (r & 7)) << 4))
                              : ~0u;
        if (idx < kItems && grow < rows_total) {
          const int si = grow / G, g = grow - si * G;
          const int sb = s_seq[si - si_lo];
          if (sb >= 0)
            v[u] = __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) +
                                                        ((size_t)sb * p.num_q_heads + h * G + g) *
                                                            D) +
                         c);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u)
        if (off[u] != ~0u) *reinterpret_cast<uint4*>(sQ + off[u]) = v[u];
    }
    tc::fence_proxy_async_smem();  // the tensor core reads what the threads wrote
    mbar_arrive(smem_addr(q_full));
  }

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    // K(0), then V(j) and K(j + 1) for each j: the order in which the MMA warp frees
    // their stages.  Lane i < kBlocksPerTile holds the id of a tile's i-th block; the ids
    // of the tile after next are loaded while the current tiles are issued.
    const uint64_t keep = l2_policy_evict_last();  // the prefix is re-read by other CTAs
    auto tile_ids = [&](int j) {
      const int bi = (kv_begin + j * BN) / BS + lane;
      int id = -1;
      if (j < n_kv && lane < C::kBlocksPerTile && bi < nblk && bi * BS < kv_end) {
        id = __ldg(p.prefix_blocks + bi);
        if (id < 0 || id >= p.num_blocks) {
          flag_status(p.status, PA_STATUS_BAD_BLOCK);
          id = -1;
        }
      }
      return id;
    };
    auto load_tile = [&](const CUtensorMap* tm, uint8_t* dst, uint64_t* full, int id) {
      if (lane == 0) mbar_arrive_expect_tx(smem_addr(full), C::kKBytes);
#pragma unroll
      for (int i = 0; i < C::kBlocksPerTile; ++i) {
        const int idi = __shfl_sync(~0u, id, i);
        if (lane == 0) {
          // a bad block id reads a box that lies wholly outside the tensor: zeros
          const int y = idi < 0 ? -BS : (idi * p.num_kv_heads + h) * BS;
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb)
            tma_load_2d(smem_addr(dst + hb * C::kKvHalfBytes + i * BS * 128), tm, hb * 64, y,
                        smem_addr(full), keep);
        }
      }
    };
    int id_cur = tile_ids(0), id_next = tile_ids(1);
    if (n_kv > 0) {
      if (!mbar_wait(smem_addr(k_empty), 1)) ok = false;
      else load_tile(&tmk, sK, k_full, id_cur);
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const int sv = j % SV;
      if (!mbar_wait(smem_addr(v_empty + sv), ((j / SV) & 1) ^ 1)) { ok = false; break; }
      load_tile(&tmv, sV + sv * C::kKBytes, v_full + sv, id_cur);
      if (j + 1 < n_kv) {
        const int sk = (j + 1) % SK;
        if (!mbar_wait(smem_addr(k_empty + sk), (((j + 1) / SK) & 1) ^ 1)) { ok = false; break; }
        load_tile(&tmk, sK + sk * C::kKBytes, k_full + sk, id_next);
      }
      id_cur = id_next;
      id_next = tile_ids(j + 2);
    }
    if (!ok && lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    // PV_A(j), S_A(j+1), PV_B(j), S_B(j+1), ... as in the chunked-prefill kernel.  The
    // whole warp runs the loop (waits included, so that it never diverges) and one elected
    // lane issues each MMA and commit: few instructions per MMA for a warp that shares its
    // scheduler with two softmax warps.
    {
      auto wait_w = [&](uint64_t* bar, uint32_t parity) {
        return __all_sync(~0u, mbar_wait(smem_addr(bar), parity));
      };
      const uint32_t id_s = tc::idesc_f16(SpFmt<T>::v, C::BM, BN, false, false);
      const uint32_t id_o = tc::idesc_f16(SpFmt<T>::v, C::BM, D, false, true);
      // descriptors of each operand's first k-step and first stage, advanced by constant
      // offsets
      const uint64_t dq0 = tc::smem_desc_sw128(smem_addr(sQ), 16, 1024);
      const uint64_t dk0 = tc::smem_desc_sw128(smem_addr(sK), 16, 1024);
      const uint64_t dv0 = tc::smem_desc_sw128(smem_addr(sV), C::kKvHalfBytes, 1024);
      auto issue_s = [&](int x, int s) {
        const uint32_t tS = tmem + x * BN;
        const uint64_t dq = tc::desc_advance(dq0, x * C::kQBytes);
        const uint64_t dk = tc::desc_advance(dk0, s * C::kKBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          tc::mma_ss_warp<false>(tS, tc::desc_advance(dq, (kk >> 2) * C::kQHalfBytes + koff),
                                 tc::desc_advance(dk, (kk >> 2) * C::kKvHalfBytes + koff), id_s,
                                 kk > 0);
        }
        tc::commit_warp<false>(smem_addr(s_full + x));
      };
      auto issue_pv = [&](int x, int j, int s) -> bool {
        if (!wait_w(p_full + x, j & 1)) return false;
        tc::fence_after_sync();
        const uint32_t tP = tmem + x * BN;
        const uint32_t tO = tmem + NT * BN + x * D;
        const uint64_t dv = tc::desc_advance(dv0, s * C::kKBytes);
        if constexpr (SpFmt<T>::v == 0) {
          // P: tokens 2c and 2c + 1 in column c
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks)
            tc::mma_ts_warp<false>(tO, tP + 8 * ks, tc::desc_advance(dv, ks * 16 * 128), id_o,
                                   j > 0 || ks > 0);
        } else {
          // P of tokens 32k .. 32k+31: hi terms in columns 32k .. 32k+15, lo terms in the next 16
#pragma unroll
          for (int ks = 0; ks < BN / 16; ++ks) {
            const uint32_t col = 32 * (ks >> 1) + 8 * (ks & 1);
            const uint64_t bdesc = tc::desc_advance(dv, ks * 16 * 128);
            tc::mma_ts_warp<false>(tO, tP + col, bdesc, id_o, j > 0 || ks > 0);
            tc::mma_ts_warp<false>(tO, tP + col + 16, bdesc, id_o, true);
          }
        }
        tc::commit_warp<false>(smem_addr(pv_done + x));
        return true;
      };
      if (n_kv > 0 && (!wait_w(q_full, 0) || !wait_w(k_full, 0))) ok = false;
      if (ok && n_kv > 0) {
        tc::fence_after_sync();
#pragma unroll
        for (int x = 0; x < NT; ++x)
          if (valid[x]) issue_s(x, 0);
        tc::commit_warp<false>(smem_addr(k_empty));  // K(0) is read by these alone
      }
      // V stage of step j and K stage of step j + 1, with their phase parities, without
      // divisions
      int sv = 0, sk1 = SK > 1 ? 1 : 0;
      uint32_t vpar = 0, kpar1 = SK > 1 ? 0 : 1;
      for (int j = 0; j < n_kv && ok; ++j) {
        bool v_ready = false, k_ready = false;
#pragma unroll
        for (int x = 0; x < NT; ++x) {
          if (!valid[x]) continue;
          if (!v_ready) {
            if (!wait_w(v_full + sv, vpar)) { ok = false; break; }
            tc::fence_after_sync();
            v_ready = true;
          }
          if (!issue_pv(x, j, sv)) { ok = false; break; }
          if (j + 1 < n_kv) {
            if (!k_ready) {
              if (!wait_w(k_full + sk1, kpar1)) { ok = false; break; }
              tc::fence_after_sync();
              k_ready = true;
            }
            issue_s(x, sk1);
          }
        }
        if (!ok) break;
        tc::commit_warp<false>(smem_addr(v_empty + sv));                 // V(j)
        if (j + 1 < n_kv) tc::commit_warp<false>(smem_addr(k_empty + sk1));  // K(j + 1)
        if (++sv == SV) { sv = 0; vpar ^= 1; }
        if (++sk1 == SK) { sk1 = 0; kpar1 ^= 1; }
      }
      if (!ok && lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------- softmax / partial output (one WG per tile) -------------------------
    const int x = (warp - 4) >> 2;
    const int r = (threadIdx.x - 128) & 127;
    const uint32_t lane_bits = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + lane_bits + x * BN;
    const uint32_t tO = tmem + lane_bits + NT * BN + x * D;
    const bool tile_valid = x == 0 ? valid[0] : valid[NT - 1];
    const float sc = p.scale_log2;
    float m = kNegInf, l = 0.f;
    for (int j = 0; j < n_kv && tile_valid; ++j) {
      if (!mbar_wait(smem_addr(s_full + x), j & 1)) { ok = false; break; }
      tc::fence_after_sync();
      const int kp0 = kv_begin + j * BN;
      const bool full = kp0 + BN <= kv_end;
      // The row is processed in 32-column chunks by loops that are not unrolled: one
      // chunk's code instead of four keeps the step's instructions within the instruction
      // cache (unrolled, each step refetched most of them).
      // Row maximum over the visible positions; on whole tiles with a positive scale the
      // raw scores are compared and the maximum scaled once.
      static_assert(BN == 128, "a 128-column row");
      float mx = kNegInf;
      if (full && sc > 0.f) {
#pragma unroll 1
        for (int k = 0; k < BN / 32; ++k) {
          float a[32];
          tc::tmem_ld32(tS + 32 * k, a);
          tc::tmem_wait_ld();
          float r0 = a[0], r1 = a[1];
#pragma unroll
          for (int i = 2; i < 32; i += 2) {
            r0 = fmaxf(r0, a[i]);
            r1 = fmaxf(r1, a[i + 1]);
          }
          mx = fmaxf(mx, fmaxf(r0, r1));
        }
        mx *= sc;
      } else {
#pragma unroll 1
        for (int k = 0; k < BN / 32; ++k) {
          float a[32];
          tc::tmem_ld32(tS + 32 * k, a);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i)
            mx = fmaxf(mx, kp0 + 32 * k + i < kv_end ? a[i] * sc : kNegInf);
        }
      }
      const bool need = mx > m + kRescaleThreshold;
      const float alpha = need ? fast_exp2(m - mx) : 1.f;
      if (need) m = mx;
      // P = 2^(scale * S - m) over S's own columns: for fp16, one term, tokens 32k .. 32k+31
      // in columns 16k .. 16k+15 (already read); for bf16, hi + lo terms in columns
      // 32k .. 32k+31.
      constexpr bool wide = SpFmt<T>::v == 1;
      float sum = 0.f;
#pragma unroll 1
      for (int k = 0; k < BN / 32; ++k) {
        float a[32];
        tc::tmem_ld32(tS + 32 * k, a);
        tc::tmem_wait_ld();
        const int c0 = 32 * k;
        if (full) {
          const uint64_t sc2 = f2(sc, sc), negm2 = f2(-m, -m);
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            float t0, t1;
            f2_split(f2_fma(f2(a[2 * i], a[2 * i + 1]), sc2, negm2), t0, t1);
            a[2 * i] = fast_exp2(t0);
            a[2 * i + 1] = fast_exp2(t1);
          }
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i)
            a[i] = kp0 + c0 + i < kv_end ? fast_exp2(fmaf(a[i], sc, -m)) : 0.f;
        }
        float s2[2] = {0.f, 0.f};
        if constexpr (!wide) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            s2[i & 1] += a[2 * i] + a[2 * i + 1];
            pk[i] = Mma<__half>::pack(a[2 * i], a[2 * i + 1]);
          }
          tc::tmem_st16(tS + 16 * k, pk);
        } else {
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            s2[i & 1] += a[2 * i] + a[2 * i + 1];
            hi[i] = Mma<T>::pack_split(a[2 * i], a[2 * i + 1], lo[i]);
          }
          tc::tmem_st16(tS + c0, hi);
          tc::tmem_st16(tS + c0 + 16, lo);
        }
        sum += s2[0] + s2[1];
      }
      l = l * alpha + sum;
      if (j >= 1 && __any_sync(~0u, need)) {
        if (!mbar_wait(smem_addr(pv_done + x), (j - 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
#pragma unroll 1
        for (int c0 = 0; c0 < D; c0 += 32) {
          float o[32];
          tc::tmem_ld32(tO + c0, o);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tc::tmem_st32(tO + c0, o);
        }
      }
      tc::tmem_wait_st();
      tc::fence_before_sync();
      mbar_arrive(smem_addr(p_full + x));
    }
    griddep_wait();  // the decode plan's partial slots (part_start) are written
    // the partial of each row: (m, l) and the unnormalised O, into the sharer's slot.  O
    // goes through shared memory (this tile's query buffer, free once its last product
    // is done) 32 columns at a time so that the global stores are whole 128-byte rows.
    bool go = ok && tile_valid && n_kv > 0;
    if (go && !mbar_wait(smem_addr(pv_done + x), (n_kv - 1) & 1)) ok = go = false;
    if (__all_sync(~0u, go)) {  // warp-collective loads and shuffles below
      tc::fence_after_sync();
      const int grow = row0 + x * C::BM + r;
      const int si = grow / G, g = grow - si * G;
      const int sb = grow < rows_total ? s_seq[si - si_lo] : -1;
      float* dst = nullptr;
      if (sb >= 0) {
        const size_t row = (size_t)(p.part_start[sb] + split) * p.num_q_heads + h * G + g;
        p.part_ml[row] = make_float2(m, l);
        dst = p.part_acc + row * D;
      }
      uint8_t* stage = sQ + x * C::kQBytes + (warp & 3) * 32 * 128;  // 32 rows x 128 B
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        tc::tmem_ld32(tO + c0, o);
        tc::tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < 8; ++k)
          *reinterpret_cast<float4*>(stage + lane * 128 + ((k ^ (lane & 7)) << 4)) =
              make_float4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
        __syncwarp();
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int rw = 4 * i + (lane >> 3), k = lane & 7;
          float* d = reinterpret_cast<float*>(
              __shfl_sync(~0u, reinterpret_cast<uintptr_t>(dst), rw));
          const float4 v =
              *reinterpret_cast<const float4*>(stage + rw * 128 + ((k ^ (rw & 7)) << 4));
          if (d != nullptr) *reinterpret_cast<float4*>(d + c0 + 4 * k) = v;
        }
        __syncwarp();
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

constexpr int kMaxDev = 64;
std::mutex g_mutex;

template <typename T, int D, int BS>
int launch_t(const DecodeArgs& a, cudaStream_t stream) {
  using C = SpCfg<D, BS>;
  static bool configured[kMaxDev] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev >= kMaxDev)
    return fail(PA_ERR_CUDA, "pa_decode_shared_prefix: no usable device");
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!configured[dev]) {
      if (cudaFuncSetAttribute(shared_prefix_kernel<T, D, BS>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)C::kSmem) != cudaSuccess)
        return fail(PA_ERR_CUDA, "pa_decode_shared_prefix: shared-memory configuration failed");
      configured[dev] = true;
    }
  }
  CUtensorMap tmk, tmv;
  const int r1 = encode_cache_map(&tmk, a.k_cache, a.dtype, a.num_blocks, a.num_kv_heads,
                                  a.block_size, a.head_dim);
  const int r2 = encode_cache_map(&tmv, a.v_cache, a.dtype, a.num_blocks, a.num_kv_heads,
                                  a.block_size, a.head_dim);
  if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS)
    return fail(PA_ERR_CUDA, "pa_decode_shared_prefix: cuTensorMapEncodeTiled failed");
  SpParams p;
  p.q = a.q;
  p.sharers = a.prefix.sharers;
  p.prefix_blocks = a.prefix.prefix_blocks;
  p.part_start = a.ws.part_start;
  p.part_ml = a.ws.part_ml;
  p.part_acc = a.ws.part_acc;
  p.status = a.status;
  p.num_sharers = a.prefix.num_sharers;
  p.prefix_len = a.prefix.prefix_len;
  p.split_tokens = a.prefix.split_tokens;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.scale_log2 = a.scale * kLog2e;
  const long long rows = (long long)a.prefix.num_sharers * p.group;
  const long long pairs = (rows + C::BM * C::kTiles - 1) / (C::BM * C::kTiles);
  if (pairs > 0x7fffffffll || a.prefix.splits > 65535 || a.num_kv_heads > 65535)
    return fail(PA_ERR_UNSUPPORTED, "pa_decode_shared_prefix: grid too large");
  const cudaError_t e =
      launch_pdl(shared_prefix_kernel<T, D, BS>,
                 dim3((unsigned)pairs, a.prefix.splits, a.num_kv_heads), dim3(C::kThreads),
                 C::kSmem, stream, tmk, tmv, p);
  if (e != cudaSuccess)
    return fail(PA_ERR_CUDA, "pa_decode_shared_prefix: %s", cudaGetErrorString(e));
  return PA_OK;
}

template <typename T>
int dispatch(const DecodeArgs& a, cudaStream_t stream) {
  if (a.head_dim == 128 && a.block_size == 16) return launch_t<T, 128, 16>(a, stream);
  if (a.head_dim == 128 && a.block_size == 32) return launch_t<T, 128, 32>(a, stream);
  if (a.head_dim == 64 && a.block_size == 16) return launch_t<T, 64, 16>(a, stream);
  if (a.head_dim == 64 && a.block_size == 32) return launch_t<T, 64, 32>(a, stream);
  return fail(PA_ERR_UNSUPPORTED, "pa_decode_shared_prefix: head_dim %d / block_size %d",
              a.head_dim, a.block_size);
}

}  // namespace

int launch_shared_prefix(const DecodeArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? dispatch<__nv_bfloat16>(a, stream) : dispatch<__half>(a, stream);
}

}  // namespace pa
