// Paged decode attention (one query token per sequence) for sm_103a.
//
// Three launches per call on the caller's stream, chained with programmatic dependent
// launch so that each one's set-up overlaps the previous one:
//   1. plan   -- one CTA reads the context lengths, picks the split-KV partition size so
//                that about kTargetUnits (partition, KV head) units exist, and writes the
//                partition list sorted largest first (longest-processing-time order, so
//                the dynamic scheduler below ends with the smallest units).  It also
//                zeroes the outputs of empty contexts and lists the sequences whose
//                partials need merging.
//   2. attend -- a persistent kernel, one CTA per SM.  Each CTA holds kPairs pairs of
//                warps; in a pair a producer warp grabs units from a global counter,
//                reads the unit's block-table entries, and streams every (block, KV
//                head) K and V tile into a ring of shared-memory stages with TMA; the
//                consumer warp runs q.K^T and P.V on the tensor cores (mma.sync
//                m16n8k16) with an online softmax: for groups of up to 8 rows the
//                products are taken transposed (tokens or dimensions as M, the group's
//                rows as N = 8), larger groups are padded to 16 rows.
//                A unit covering a whole context writes the normalised output; the
//                others write an fp32 partial (running max, sum, unnormalised output).
//   3. merge  -- one warp per (sequence, query head) of a listed sequence merges its
//                partials by log-sum-exp rescaling.  (Merging inside the attention
//                kernel, by whichever warp finished last, stalled that warp's pipeline
//                on a device-wide fence and an atomic round trip per partition, which
//                cost more than this launch.)
// fp32 caches take a CUDA-core variant of step 2 (tensor cores have no fp32 input path
// that meets an fp32 tolerance).
//
// The decode is bound by HBM: every context token's K and V row is read once and each
// byte feeds ~1 (MHA) to ~8 (group of 8) flops, far below the ridge point.  The design
// therefore aims at bytes in flight (up to 192 KiB of TMA copies per SM) and keeps the
// per-tile instruction count small.
#include <algorithm>
#include <climits>
#include <mutex>

#include "pa_device.cuh"
#include "pa_internal.h"
#include "pa_launch.h"

namespace pa {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
// The running maximum is only moved when a tile's maximum exceeds it by more than this
// many powers of two; in between, probabilities up to 2^8 are accumulated, which fp32
// sums and 16-bit hi/lo splits of P represent without loss of accuracy.
constexpr float kRescaleThreshold = 8.0f;
constexpr float kNegInf = -__builtin_huge_valf();

struct DecodeParams {
  const void* q;
  void* out;
  const int32_t* block_tables;
  const int32_t* context_lens;
  DecodeWorkspace ws;
  int32_t* status;
  int max_blocks, ctx_cap, num_seqs, num_q_heads, num_kv_heads, group, num_blocks;
  int out_f32;     // fp32 output from 16-bit inputs
  int out_bytes;   // bytes per output element
  int out_bf16;    // output is bf16
  float scale_log2;
  // the caches, for L2 prefetches of the first partitions' K/V while the plan is built
  const void* k_cache;
  const void* v_cache;
  long long prefetch_bytes;  // at most this many bytes prefetched (0: none)
  // The attention kernel waits for the plan through the workspace flag (header[5], set
  // by the plan once its list is written) rather than through the launch dependency, and
  // for the kernel launched just before it (the shared prefix's) only before it exits.
  int plan_flag;
  int forced_psz;  // partition size set by the caller (tokens), 0: chosen from the batch
  // With a shared prefix and `early` set, the producers start on the plan's first units
  // before the plan is done (see early_records): the sharer list and the prefix's
  // geometry, as the plan has them.
  const int32_t* sharers;
  int num_sharers, prefix_len, prefix_splits, max_own_parts;
  int early;
};

// A unit as the producer hands it to its consumer.
struct UnitDesc {
  int b, h, tok0, ntok, nparts, part_idx, part_start, valid;
};

__device__ __forceinline__ int clamp_ctx(int c, int cap) { return c < 0 ? 0 : (c > cap ? cap : c); }

// Tokens per split-KV partition for a batch of `total` context tokens: about kTargetUnits
// (partition, KV head) units, whole blocks, within [kMinPartBlocks, kMaxPartBlocks] blocks.
// The plan kernel sets the partitions with it, and the attention kernel recomputes it to
// predict the plan's first units.
// A positive `forced` (whole blocks, set only by the testing entry point) replaces the choice.
__device__ __forceinline__ int partition_tokens(long long total, int num_kv_heads, int block_size,
                                                int forced) {
  if (forced > 0) return forced;
  long long want = (total * num_kv_heads + kTargetUnits - 1) / kTargetUnits;
  want = (want + block_size - 1) / block_size * block_size;
  want = max(want, (long long)kMinPartBlocks * block_size);
  want = min(want, (long long)kMaxPartBlocks * block_size);
  return (int)want;
}

// The same with a shared prefix: partitions long enough that every sharer's partials (its
// `max_own_parts` own partitions at most, beside its prefix splits) are merged in one
// round.  `tmax` is the longest own context (past the prefix) of a sharer.
__device__ __forceinline__ int batch_partition_tokens(long long total, int tmax,
                                                      int num_kv_heads, int block_size,
                                                      int forced, int num_sharers,
                                                      int max_own_parts) {
  int psz = partition_tokens(total, num_kv_heads, block_size, forced);
  if (forced <= 0 && num_sharers > 0 && max_own_parts > 0 && tmax > psz) {
    long long need = (tmax + max_own_parts - 1) / max_own_parts;
    need = (need + block_size - 1) / block_size * block_size;
    psz = (int)max((long long)psz, min(need, (long long)kMaxPartBlocks * block_size));
  }
  return psz;
}

// ----------------------------------------------------------------------------------
// 1. plan
// ----------------------------------------------------------------------------------

// Claims one slot of counters[key] for every lane with key >= 0, with one shared-memory
// atomic per distinct key in the warp; the lanes of a key take consecutive slots in lane
// order.  Returns the lane's slot (meaningless for key < 0).  All 32 lanes must call it.
__device__ __forceinline__ int warp_claim(int* counters, int key, int lane) {
  const unsigned grp = __match_any_sync(~0u, key);
  const int leader = __ffs(grp) - 1;
  int base = 0;
  if (key >= 0 && lane == leader) base = atomicAdd(counters + key, __popc(grp));
  base = __shfl_sync(~0u, base, leader);
  return base + __popc(grp & ((1u << lane) - 1));
}

__global__ void __launch_bounds__(1024, 1) decode_plan_kernel(const int32_t* __restrict__ context_lens,
                                                           int num_seqs, int ctx_cap,
                                                           int num_kv_heads, int block_size,
                                                           DecodeWorkspace ws, int32_t* status,
                                                           int4* out, int out_row_vec16,
                                                           PrefixPlan pre, int wait_late,
                                                           int forced_psz, int early) {
  // wait_late: the previous kernel on the stream writes nothing this kernel reads or
  // writes; it is waited for only at the end, so that the work list is built meanwhile
  // and the next kernel still starts after both (lengths are read through L2)
  if (!wait_late) griddep_wait();
  // with a shared prefix the attention kernel waits for the flag this kernel sets at its
  // end: cleared before the kernels after this one may launch, like the counter of the
  // units it takes before that flag (`early`: the full partitions, which head the list)
  if (pre.num_sharers > 0 && threadIdx.x == 0) {
    ws.header[5] = 0;
    if (early) ws.header[6] = 0;
    __threadfence();
  }
  griddep_launch_dependents();
  __shared__ long long s_sum[32];
  __shared__ int s_smax[32];
  __shared__ int s_off[32], s_foff[32];
  __shared__ int s_ftotal;
  __shared__ int s_hist[kMaxPartBlocks + 2];
  __shared__ int s_psz, s_total, s_units, s_nmerge;
  // each sequence's own context (past a shared prefix), read once from memory: the later
  // passes take it from here (each thread reads back only what it wrote)
  constexpr int kSufCache = 4096;
  __shared__ int s_suf[kSufCache];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5, nwarps = blockDim.x >> 5;
  const int per = (num_seqs + blockDim.x - 1) / blockDim.x;
  const int b0 = min(num_seqs, tid * per), b1 = min(num_seqs, b0 + per);
  // the thread's first context length, loaded while the sharer flags are set up (an input
  // of the call: no kernel before this one writes it)
  const int c_first = b0 < b1 ? __ldcg(context_lens + b0) : 0;

  // sequences reading a shared prefix start their own partitions after it and keep
  // pre.splits partial slots, ahead of those, for the prefix's partials.  Which sequences
  // they are is read in every pass below: from shared memory for batches of up to
  // kSufCache sequences, from the workspace beyond.
  __shared__ unsigned char s_flag[kSufCache];
  const bool flags_shared = num_seqs <= kSufCache;
  if (pre.num_sharers > 0) {
    for (int b = tid; b < num_seqs; b += blockDim.x) {
      if (flags_shared) s_flag[b] = 0;
      else ws.seq_flags[b] = 0;
    }
    __syncthreads();
    for (int i = tid; i < pre.num_sharers; i += blockDim.x) {
      const int sb = pre.sharers[i];
      if (sb >= 0 && sb < num_seqs) {
        if (flags_shared) s_flag[sb] = 1;
        else ws.seq_flags[sb] = 1;
      } else {
        flag_status(status, PA_STATUS_BAD_CONTEXT);
      }
    }
    __syncthreads();
  }
  auto sharer = [&](int b) {
    return pre.num_sharers > 0 && (flags_shared ? s_flag[b] != 0 : ws.seq_flags[b] != 0);
  };
  auto start_of = [&](int b) { return sharer(b) ? pre.prefix_len : 0; };
  auto reserved_of = [&](int b) { return sharer(b) ? pre.splits : 0; };

  long long sum = 0;
  int smax = 0;  // the longest own context of a sequence reading the shared prefix
  for (int b = b0; b < b1; ++b) {
    const int c = b == b0 ? c_first : __ldcg(context_lens + b);
    if (c < 0 || c > ctx_cap) flag_status(status, PA_STATUS_BAD_CONTEXT);
    const int cc = clamp_ctx(c, ctx_cap), st = start_of(b);
    if (cc < st) flag_status(status, PA_STATUS_BAD_CONTEXT);
    sum += max(0, cc - st);
    if (st > 0) smax = max(smax, cc - st);
    if (b < kSufCache) s_suf[b] = max(0, cc - st);
    if (cc == 0 && reserved_of(b) == 0)  // an empty context attends to nothing: zeros
      for (int i = 0; i < out_row_vec16; ++i) out[(size_t)b * out_row_vec16 + i] = make_int4(0, 0, 0, 0);
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    sum += __shfl_xor_sync(~0u, sum, o);
    smax = max(smax, __shfl_xor_sync(~0u, smax, o));
  }
  if (lane == 0) {
    s_sum[wid] = sum;
    s_smax[wid] = smax;
  }
  for (int i = tid; i < kMaxPartBlocks + 2; i += blockDim.x) s_hist[i] = 0;
  if (tid == 0) s_nmerge = 0;
  __syncthreads();
  if (wid == 0) {
    long long total = lane < nwarps ? s_sum[lane] : 0;
    int tmax = lane < nwarps ? s_smax[lane] : 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      total += __shfl_xor_sync(~0u, total, o);
      tmax = max(tmax, __shfl_xor_sync(~0u, tmax, o));
    }
    if (lane == 0)
      s_psz = batch_partition_tokens(total, tmax, num_kv_heads, block_size, forced_psz,
                                     pre.num_sharers, pre.max_own_parts);
  }
  __syncthreads();
  const int psz = s_psz, bpp = psz / block_size;
  auto suffix_of = [&](int b) {
    return b < kSufCache ? s_suf[b]
                         : max(0, clamp_ctx(__ldcg(context_lens + b), ctx_cap) - start_of(b));
  };

  // Counting pass.  Every lane runs `per` iterations (so that whole warps meet in the
  // shuffles and matches), and shared counters are bumped once per warp and distinct key.
  auto tail_bucket = [&](int c, int np) {
    return np > 0 ? (c - (np - 1) * psz + block_size - 1) / block_size : -1;
  };
  int local = 0, full = 0;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    int c = 0, np = 0, rs = 0;
    if (b < b1) {
      c = suffix_of(b);
      np = (c + psz - 1) / psz;
      rs = reserved_of(b);
    }
    local += np + rs;
    // several partials, or any for a shared prefix: the merge kernel combines them (the
    // list's order does not matter, each sequence is merged on its own)
    const bool merge = np + rs > 1 || rs > 0;
    const int m = warp_claim(&s_nmerge, merge ? 0 : -1, lane);
    if (merge) ws.merge_seqs[m] = b;
    warp_claim(s_hist, tail_bucket(c, np), lane);
    full += np > 1 ? np - 1 : 0;
  }
  // full partitions take the first slots of the list in sequence order (so that the
  // attention kernel can predict them): each thread's offset is an exclusive scan of the
  // full-partition counts over threads, which own consecutive sequences
  const int flocal = full;
  int fincl = flocal;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(~0u, fincl, o);
    if (lane >= o) fincl += v;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) full += __shfl_xor_sync(~0u, full, o);
  if (lane == 0 && full > 0) atomicAdd(&s_hist[bpp], full);
  int incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) {
    s_off[wid] = incl;
    s_foff[wid] = fincl;
  }
  __syncthreads();
  if (wid == 0) {
    const int v = lane < nwarps ? s_off[lane] : 0;
    const int fv = lane < nwarps ? s_foff[lane] : 0;
    int iv = v, ifv = fv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(~0u, iv, o);
      const int ft = __shfl_up_sync(~0u, ifv, o);
      if (lane >= o) {
        iv += t;
        ifv += ft;
      }
    }
    if (lane < nwarps) {
      s_off[lane] = iv - v;
      s_foff[lane] = ifv - fv;
    }
    if (lane == 31) {
      s_total = iv;
      s_ftotal = ifv;
    }
  }
  __syncthreads();
  int run = s_off[wid] + incl - local;
  for (int b = b0; b < b1; ++b) {
    ws.part_start[b] = run;
    run += (suffix_of(b) + psz - 1) / psz + reserved_of(b);
  }
  if (tid == 0) ws.part_start[num_seqs] = s_total;
  if (wid == 0) {
    // bucket offsets, largest partitions first: an exclusive scan of s_hist[bpp .. 1]
    // by one warp, each lane owning kMaxPartBlocks / 32 consecutive buckets
    constexpr int per = kMaxPartBlocks / 32;
    int v[per], run = 0;
#pragma unroll
    for (int k = 0; k < per; ++k) {
      const int bucket = bpp - (lane * per + k);
      v[k] = bucket >= 1 ? s_hist[bucket] : 0;
      run += v[k];
    }
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int t = __shfl_up_sync(~0u, incl, o);
      if (lane >= o) incl += t;
    }
    int off = incl - run;
#pragma unroll
    for (int k = 0; k < per; ++k) {
      const int bucket = bpp - (lane * per + k);
      if (bucket >= 1) s_hist[bucket] = off;
      off += v[k];
    }
    if (lane == 31) s_units = incl;  // partitions with a K/V range of their own
    // the largest bucket (offset 0) starts with every full partition, placed below; last
    // partitions of that size are claimed after them
    if (lane == 0) s_hist[bpp] += s_ftotal;
  }
  __syncthreads();
  // Placement pass: a sequence's np - 1 full partitions take consecutive slots after those
  // of the sequences before it, its last one a slot of its own bucket.
  run = s_off[wid] + incl - local;
  int frun = s_foff[wid] + fincl - flocal;
  for (int i = 0; i < per; ++i) {
    const int b = b0 + i;
    int c = 0, st = 0, rs = 0, np = 0;
    if (b < b1) {
      c = suffix_of(b);
      st = start_of(b);
      rs = reserved_of(b);
      np = (c + psz - 1) / psz;
    }
    const int fbase = frun;
    frun += np > 1 ? np - 1 : 0;
    const int tslot = warp_claim(s_hist, tail_bucket(c, np), lane);
    for (int p = 0; p < np; ++p) {
      const int ntok = min(psz, c - p * psz);
      const int slot = p + 1 < np ? fbase + p : tslot;
      PartRec r;
      r.b = b;
      r.p = rs + p;
      r.tok0 = st + p * psz;
      r.ntok = ntok;
      r.part_start = run;
      r.nparts = np + rs;
      r.pad0 = r.pad1 = 0;
      ws.parts[slot] = r;
    }
    run += np + rs;
  }
  if (tid == 0) {
    // with `early`, the attention kernel has taken the full partitions by a counter of its
    // own: this list's counter starts past them
    ws.header[0] = early ? s_ftotal * num_kv_heads : 0;
    ws.header[1] = s_units * num_kv_heads;
    ws.header[2] = psz;
    ws.header[3] = s_total;
    ws.header[4] = s_nmerge;
  }
  if (wait_late) griddep_wait();
  if (pre.num_sharers > 0) {
    __threadfence();  // every thread's writes, before the flag
    __syncthreads();
    if (tid == 0) atomicExch(ws.header + 5, 1);
  }
}

// A unit is (partition, KV head): unit u is partition u / H_kv for KV head u % H_kv.
__device__ __forceinline__ PartRec load_part(const DecodeParams& p, int u) {
  const int4* src = reinterpret_cast<const int4*>(p.ws.parts + u / p.num_kv_heads);
  const int4 a = __ldcg(src), c = __ldcg(src + 1);  // written by the plan kernel
  PartRec r;
  r.b = a.x; r.p = a.y; r.tok0 = a.z; r.ntok = a.w;
  r.part_start = c.x; r.nparts = c.y; r.pad0 = c.z; r.pad1 = c.w;
  return r;
}

__device__ __forceinline__ UnitDesc describe_unit(const PartRec& r, int u, int num_kv_heads) {
  UnitDesc d;
  d.b = r.b;
  d.h = u % num_kv_heads;
  d.tok0 = r.tok0;
  d.ntok = r.ntok;
  d.nparts = r.nparts;
  d.part_idx = r.part_start + r.p;
  d.part_start = r.part_start;
  d.valid = 1;
  return d;
}

// Combines two (max, sum) pairs of the same row in log2 units.
__device__ __forceinline__ void combine_ml(float& m, float& l, float m2, float l2) {
  const float mx = fmaxf(m, m2);
  if (mx == kNegInf) return;  // both empty
  l = l * fast_exp2(m - mx) + l2 * fast_exp2(m2 - mx);
  m = mx;
}

constexpr int kMaxGroup = 16;
// Sequences with up to this many partitions are merged with one round of loads (D = 64;
// six for D = 128, within the merge kernel's 64 registers a thread).
constexpr int kMergeOneRound = 8;
// the partials merge_row takes in one round for head dim D
constexpr int merge_one_round(int D) { return D == 128 ? 6 : kMergeOneRound; }
// Merge grid: CTAs of 256 threads per SM (at most 64 registers a thread, so that four
// fit in the register file).
constexpr int kMergeCtasPerSm = 4;

// Merges the partials of one (sequence, query head):
// out = sum_p 2^(m_p - M) acc_p / sum_p 2^(m_p - M) l_p with M = max_p m_p.  Run by one
// warp; each lane owns D/32 consecutive columns.  Up to kMergeOneRound partitions, every
// (max, sum) pair and partial output row is loaded in one round; beyond that, two
// dependent rounds: the (max, sum) of every partition, then every partial output row, all
// in flight together.  The partials were written by the previous kernel and are read
// through L2.
// Loads C (4 or 2) consecutive floats through L2.
template <int C>
__device__ __forceinline__ void ldcg_vec(const float* ptr, float* dst) {
  if constexpr (C == 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(ptr));
    dst[0] = v.x; dst[1] = v.y; dst[2] = v.z; dst[3] = v.w;
  } else {
    const float2 v = __ldcg(reinterpret_cast<const float2*>(ptr));
    dst[0] = v.x; dst[1] = v.y;
  }
}

template <int D, typename TO>
__device__ __forceinline__ void merge_row(const DecodeParams& p, int b, int hq, int ps, int np,
                                          TO* out, int lane) {
  constexpr int C = D / 32;
  constexpr int R = merge_one_round(D);
  const size_t hs = (size_t)p.num_q_heads;
  const float2* ml = p.ws.part_ml + (size_t)ps * hs + hq;  // stride hs per partition
  const float* src = p.ws.part_acc + ((size_t)ps * hs + hq) * D + lane * C;
  float acc[C];
#pragma unroll
  for (int c = 0; c < C; ++c) acc[c] = 0.f;
  float M = kNegInf, L = 0.f;
  if (np <= R) {
    float2 mv[R];
    float av[R][C];
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (i < np) {
        mv[i] = __ldcg(ml + i * hs);
        ldcg_vec<C>(src + (size_t)i * hs * D, av[i]);
      }
    }
#pragma unroll
    for (int i = 0; i < R; ++i)
      if (i < np) M = fmaxf(M, mv[i].x);
#pragma unroll
    for (int i = 0; i < R; ++i) {
      if (i < np) {
        const float w = fast_exp2(mv[i].x - M);
        L += w * mv[i].y;
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] += w * av[i][c];
      }
    }
  } else {
    float m_own = kNegInf;
    for (int i0 = 0; i0 < np; i0 += 32) {
      const int i = i0 + lane;
      if (i < np) {
        const float2 v = __ldcg(ml + i * hs);
        if (i0 == 0) m_own = v.x;
        combine_ml(M, L, v.x, v.y);
      }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
      const float m2 = __shfl_xor_sync(~0u, M, o);
      const float l2 = __shfl_xor_sync(~0u, L, o);
      combine_ml(M, L, m2, l2);
    }
    for (int i0 = 0; i0 < np; i0 += 32) {
      const int i = i0 + lane;
      float w = 0.f;
      if (i < np) w = fast_exp2((i0 == 0 ? m_own : __ldcg(ml + i * hs).x) - M);
      const int n = min(32, np - i0);
#pragma unroll 4
      for (int j = 0; j < n; ++j) {
        const float wj = __shfl_sync(~0u, w, j);
        float v[C];
        ldcg_vec<C>(src + (size_t)(i0 + j) * hs * D, v);
#pragma unroll
        for (int c = 0; c < C; ++c) acc[c] += wj * v[c];
      }
    }
  }
  const float inv = 1.f / L;
  TO* o = out + ((size_t)b * p.num_q_heads + hq) * D + lane * C;
#pragma unroll
  for (int c = 0; c < C; c += 2) store2(o + c, acc[c] * inv, acc[c + 1] * inv);
}

// 3. merge: one warp per (sequence, query head) of a sequence on the plan's merge list,
// in a grid that stays resident beside the attention kernel's last CTAs (warps loop when
// the list has more rows than the grid has warps).
template <int D, typename TO>
__global__ void __launch_bounds__(256, kMergeCtasPerSm) decode_merge_kernel(const DecodeParams p) {
  const int lane = threadIdx.x & 31;
  const int nw = gridDim.x * (blockDim.x >> 5);
  const int hs = p.num_q_heads;
  int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  // The merge list and partition table come from the plan kernel, which finished before
  // the attention kernel passed its own dependency wait, and so before this grid was
  // launched: a warp's first row is looked up (through L2) ahead of the wait, off the path
  // that starts when the attention kernel ends.
  const int rows = __ldcg(p.ws.header + 4) * hs;
  int b = 0, ps = 0, np = 0;
  if (r < rows) {
    b = __ldcg(p.ws.merge_seqs + r / hs);
    ps = __ldcg(p.ws.part_start + b);
    np = __ldcg(p.ws.part_start + b + 1) - ps;
  }
  griddep_wait();  // every partial of the attention kernel is written
  griddep_launch_dependents();
  while (r < rows) {
    merge_row<D, TO>(p, b, r - (r / hs) * hs, ps, np, static_cast<TO*>(p.out), lane);
    r += nw;
    if (r < rows) {
      b = __ldcg(p.ws.merge_seqs + r / hs);
      ps = __ldcg(p.ws.part_start + b);
      np = __ldcg(p.ws.part_start + b + 1) - ps;
    }
  }
}

using MergeKernel = void (*)(DecodeParams);
template <int D>
MergeKernel merge_kernel_for(pa_dtype out) {
  if (out == PA_F32) return decode_merge_kernel<D, float>;
  if (out == PA_BF16) return decode_merge_kernel<D, __nv_bfloat16>;
  return decode_merge_kernel<D, __half>;
}

// ----------------------------------------------------------------------------------
// 2a. attend: TMA + tensor cores (fp16 / bf16)
// ----------------------------------------------------------------------------------
// Four producer/consumer warp pairs per SM, each with a 48 KiB ring, 192 KiB in all.  Three
// pairs of 64 KiB come within 0.3-0.6% on batches streamed from HBM but lose 18% where the
// consumers' arithmetic sets the pace (K/V that L2 holds because many sequences read it);
// two pairs of 96 KiB lose everywhere.
template <int D, int BS, int EB>
struct MmaCfg {
  static constexpr int kPairs = 4;
  static constexpr int kBoxBytes = BS * 128;             // BS rows x 64 elements (128 B)
  static constexpr int kHalves = D / 64;                 // boxes per K (or V) tile
  static constexpr int kTileBytes = kHalves * kBoxBytes;  // one K or V tile
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kRingBytesPerPair = 48 * 1024;
  static constexpr int kStages =
      kRingBytesPerPair / kStageBytes > 8 ? 8 : kRingBytesPerPair / kStageBytes;
  static constexpr int kThreads = 2 * kPairs * 32;
  static constexpr int kBars = 2 * kPairs * kStages + 4 * kPairs;

  __host__ __device__ static size_t qstride(int group) {
    return ((size_t)group * D * EB + 127) / 128 * 128;
  }
  static size_t smem_bytes(int group) {
    return 1024 + (size_t)kPairs * kStages * kStageBytes + kPairs * 2 * qstride(group) + 128 +
           kBars * 8 + kPairs * 2 * sizeof(UnitDesc);
  }
};

// Consumer warp for query groups of up to 8 rows.  The products are taken transposed, so
// that a tile's 16 tokens (or 16 dimensions) are the MMA's M and the group's rows its
// N = 8 (m16n8k16), half the MMAs of the group padded to 16 rows:
//   S^T[tok][row]  = K[tok][:] . Q[row][:]            A = K rows, B = Q^T
//   O^T[dim][row] += V^T[dim][tok] . P^T[tok][row]    A = V^T (transposed ldmatrix),
//                                                      B = P^T (movmatrix of S^T's layout)
// Lane l holds rows 2 (l % 4) and 2 (l % 4) + 1, and tokens / dimensions l / 4 and
// l / 4 + 8 of each 16-wide tile.  Rows >= G are zero queries and are never written.
template <typename T, int D, int BS, typename C>
__device__ __forceinline__ void consume_t(const DecodeParams& p, UnitDesc* mydesc,
                                          uint8_t* myq, uint32_t qstride, uint64_t* qfull,
                                          uint64_t* qempty, uint64_t* full, uint64_t* empty,
                                          uint8_t* mystages, uint32_t zero_addr, int lane) {
  using M = Mma<T>;
  constexpr int S = C::kStages;
  constexpr int MT = BS / 16;  // 16-token tiles of S^T per K/V tile
  constexpr int KS = D / 16;   // k-steps of K.q
  constexpr int DT = D / 16;   // 16-dimension tiles of O^T
  const int G = p.group;
  const int q4 = lane & 3, g8 = lane >> 2;
  uint32_t tile_it = 0, q_it = 0;
  for (;;) {
    const int qs = q_it & 1;
    if (!mbar_wait(smem_addr(qfull + qs), (q_it >> 1) & 1)) {
      if (lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
      return;
    }
    const UnitDesc d = mydesc[qs];
    if (!d.valid) return;

    // Q^T as B fragments: qb[k][0] = Q[row l/4][dims 16k + 2 (l%4), +1], qb[k][1] the same
    // 8 dims on; one ldmatrix x4 reads two k-steps (16-byte chunks 2k .. 2k + 3)
    uint32_t qb[KS][2];
    {
      const int r = lane & 7, i = lane >> 3;
      const uint32_t rowbase = smem_addr(myq + qs * qstride) + r * (D * sizeof(T));
#pragma unroll
      for (int kk = 0; kk < KS; kk += 2) {
        const uint32_t addr = r < G ? rowbase + (2 * kk + i) * 16 : zero_addr;
        ldsm_x4(addr, qb[kk][0], qb[kk][1], qb[kk + 1][0], qb[kk + 1][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(qempty + qs));
    ++q_it;

    float o[DT][4];  // O^T: [dt][0] dim 16 dt + l/4, row 2 (l%4); [1] row + 1; [2], [3] dim + 8
#pragma unroll
    for (int j = 0; j < DT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float mr[2] = {kNegInf, kNegInf}, lr[2] = {0.f, 0.f};  // per row: max (log2), sum

    const int ntiles = (d.ntok + BS - 1) / BS;
    for (int t = 0; t < ntiles; ++t) {
      const int s = tile_it % S;
      if (!mbar_wait(smem_addr(full + s), (tile_it / S) & 1)) {
        if (lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
        return;
      }
      const uint32_t kbase = smem_addr(mystages + (size_t)s * C::kStageBytes);
      const uint32_t vbase = kbase + C::kTileBytes;

      // S^T[16 MT tokens x 8 rows]; even and odd k-steps in two accumulators
      float sc[MT][4];
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        float sd[4] = {0.f, 0.f, 0.f, 0.f};
        sc[mt][0] = sc[mt][1] = sc[mt][2] = sc[mt][3] = 0.f;
        // ldmatrix x4 of K rows: (tok 0-7, chunk lo), (tok 8-15, lo), (0-7, hi), (8-15, hi)
        const int tok = 16 * mt + (lane & 7) + 8 * ((lane >> 3) & 1);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const int cg = 2 * kk + (lane >> 4);
          const uint32_t addr =
              kbase + (cg >> 3) * C::kBoxBytes + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4);
          uint32_t a[4];
          ldsm_x4(addr, a[0], a[1], a[2], a[3]);
          if (kk & 1) M::run(sd, a, qb[kk][0], qb[kk][1]);
          else M::run(sc[mt], a, qb[kk][0], qb[kk][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[mt][e] += sd[e];
      }
      // scale into log2 units; tokens past the context never count
      const int limit = d.ntok - t * BS;
      float mx[2] = {kNegInf, kNegInf};
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const bool valid = 16 * mt + g8 + 8 * (e >> 1) < limit;
          sc[mt][e] = valid ? sc[mt][e] * p.scale_log2 : kNegInf;
          mx[e & 1] = fmaxf(mx[e & 1], sc[mt][e]);
        }
      }
      // a row's tokens are spread over the 8 lanes with the same l % 4
#pragma unroll
      for (int off = 4; off < 32; off <<= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(~0u, mx[0], off));
        mx[1] = fmaxf(mx[1], __shfl_xor_sync(~0u, mx[1], off));
      }
      const bool need0 = mx[0] > mr[0] + kRescaleThreshold;
      const bool need1 = mx[1] > mr[1] + kRescaleThreshold;
      if (__any_sync(~0u, need0 || need1)) {
        if (need0) {
          const float a = fast_exp2(mr[0] - mx[0]);
          mr[0] = mx[0];
          lr[0] *= a;
#pragma unroll
          for (int j = 0; j < DT; ++j) { o[j][0] *= a; o[j][2] *= a; }
        }
        if (need1) {
          const float a = fast_exp2(mr[1] - mx[1]);
          mr[1] = mx[1];
          lr[1] *= a;
#pragma unroll
          for (int j = 0; j < DT; ++j) { o[j][1] *= a; o[j][3] *= a; }
        }
      }
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          sc[mt][e] = fast_exp2(sc[mt][e] - mr[e & 1]);
          lr[e & 1] += sc[mt][e];
        }
      }
      // O^T += V^T . P^T, one 16-token k-step per S^T tile, P^T carried as hi + lo terms:
      // S^T's fragment rows are tokens, a B fragment's are rows of the group, so each
      // 8 x 8 block of packed P^T is transposed across the warp
#pragma unroll
      for (int mt = 0; mt < MT; ++mt) {
        uint32_t l0, l1;
        const uint32_t h0 = movmatrix_trans(M::pack_split(sc[mt][0], sc[mt][1], l0));
        const uint32_t h1 = movmatrix_trans(M::pack_split(sc[mt][2], sc[mt][3], l1));
        l0 = movmatrix_trans(l0);
        l1 = movmatrix_trans(l1);
        // V rows of tokens past the context may hold anything (even NaN bits) and meet
        // P = 0: clear them in the fragments of the last tile
        const int vlim = limit - 16 * mt;
        const bool tail = vlim < 16;
        const uint32_t m_lo = (2 * q4 < vlim ? 0x0000ffffu : 0u) | (2 * q4 + 1 < vlim ? 0xffff0000u : 0u);
        const uint32_t m_hi =
            (2 * q4 + 8 < vlim ? 0x0000ffffu : 0u) | (2 * q4 + 9 < vlim ? 0xffff0000u : 0u);
        // ldmatrix x4 .trans of V rows: (tok 0-7, chunk 2dt), (0-7, 2dt+1), (8-15, 2dt),
        // (8-15, 2dt+1) give the A fragments of V^T for dims 16 dt .. 16 dt + 15
        const int tok = 16 * mt + (lane & 7) + 8 * (lane >> 4);
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          const int cg = 2 * dt + ((lane >> 3) & 1);
          const uint32_t addr =
              vbase + (cg >> 3) * C::kBoxBytes + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4);
          uint32_t a[4];
          ldsm_x4_trans(addr, a[0], a[1], a[2], a[3]);
          if (tail) {
            a[0] &= m_lo;
            a[1] &= m_lo;
            a[2] &= m_hi;
            a[3] &= m_hi;
          }
          M::run(o[dt], a, h0, h1);
          M::run(o[dt], a, l0, l1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(empty + s));
      ++tile_it;
    }

#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      lr[0] += __shfl_xor_sync(~0u, lr[0], off);
      lr[1] += __shfl_xor_sync(~0u, lr[1], off);
    }
    const int hq0 = d.h * G;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int row = 2 * q4 + i;
      if (row >= G) continue;
      if (d.nparts == 1) {
        const float inv = 1.f / lr[i];
        const size_t at = ((size_t)d.b * p.num_q_heads + hq0 + row) * D + g8;
        if (p.out_f32) {
          float* out = static_cast<float*>(p.out) + at;
#pragma unroll
          for (int j = 0; j < DT; ++j) {
            out[16 * j] = o[j][i] * inv;
            out[16 * j + 8] = o[j][2 + i] * inv;
          }
        } else {
          T* out = static_cast<T*>(p.out) + at;
#pragma unroll
          for (int j = 0; j < DT; ++j) {
            store1(out + 16 * j, o[j][i] * inv);
            store1(out + 16 * j + 8, o[j][2 + i] * inv);
          }
        }
      } else {
        const size_t slot = (size_t)d.part_idx * p.num_q_heads + hq0 + row;
        float* acc = p.ws.part_acc + slot * D + g8;
#pragma unroll
        for (int j = 0; j < DT; ++j) {
          acc[16 * j] = o[j][i];
          acc[16 * j + 8] = o[j][2 + i];
        }
        if (g8 == 0) p.ws.part_ml[slot] = make_float2(mr[i], lr[i]);
      }
    }
  }
}

// Sequences up to which the attention kernel predicts the plan's first units, and the
// bytes of those units' K/V it brings into L2 meanwhile (about what HBM moves while the
// plan is built).
constexpr int kPrefetchMaxSeqs = 4096;
constexpr long long kDecodePrefetchBytes = 48ll << 20;

// While the plan is being built, brings into L2 the K/V of the first units the attention
// kernel will take: the plan puts every sequence's full partitions first, in sequence
// order, with a partition size that depends only on the clamped context lengths, so each
// CTA recomputes both from the lengths (in `scratch`, 2 * kPrefetchMaxSeqs + 64 ints of
// shared memory) and its threads spread the first prefetch_bytes of those units over the
// grid, one block of one unit at a time.  Hints only: what the kernel computes does not depend on them.  Every thread of
// the CTA calls it.
template <typename T, int D, int BS, int NT>
__device__ void prefetch_first_units(const DecodeParams& p, int* scratch) {
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = p.num_seqs, hkv = p.num_kv_heads;
  int* s_c = scratch;                          // clamped context length of each sequence
  int* s_f = scratch + kPrefetchMaxSeqs;       // its first full partition's index
  long long* s_red = reinterpret_cast<long long*>(scratch + 2 * kPrefetchMaxSeqs);
  int* s_w = scratch + 2 * kPrefetchMaxSeqs + 2 * (NT / 32);
  long long tot = 0;
  for (int b = tid; b < n; b += NT) {
    const int c = clamp_ctx(__ldcg(p.context_lens + b), p.ctx_cap);
    s_c[b] = c;
    tot += c;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) tot += __shfl_xor_sync(~0u, tot, o);
  if (lane == 0) s_red[wid] = tot;
  __syncthreads();
  long long total = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) total += s_red[w];
  const int psz = partition_tokens(total, hkv, BS, p.forced_psz), bpp = psz / BS;
  auto nfull = [&](int c) { return c > psz ? (c + psz - 1) / psz - 1 : 0; };
  const int per = (n + NT - 1) / NT, b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) sum += nfull(s_c[b]);
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(~0u, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) s_w[wid] = incl;
  __syncthreads();
  int off = incl - sum, ftotal = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < wid) off += s_w[w];
    ftotal += s_w[w];
  }
  for (int b = b0; b < b1; ++b) {
    s_f[b] = off;
    off += nfull(s_c[b]);
  }
  __syncthreads();
  constexpr uint32_t kSlice = BS * D * sizeof(T);  // one block of one head, K or V
  const long long unit_bytes = 2ll * bpp * kSlice;
  const long long units = min((long long)ftotal * hkv, p.prefetch_bytes / unit_bytes);
  const T* kc = static_cast<const T*>(p.k_cache);
  const T* vc = static_cast<const T*>(p.v_cache);
  // one (unit, block) pair per thread at a time, spread over the whole grid (each SM's
  // bulk-copy engine also serves its own K/V loads)
  const long long pairs = units * bpp, stride = (long long)gridDim.x * NT;
  for (long long f = (long long)blockIdx.x * NT + tid; f < pairs; f += stride) {
    const long long u = f / bpp;
    const int i = (int)(f - u * bpp);
    const int q = (int)(u / hkv), h = (int)(u - (long long)q * hkv);
    int lo = 0, hi = n;  // the last sequence whose first full partition is <= q
    while (lo < hi) {
      const int mid = (lo + hi) >> 1;
      if (s_f[mid] <= q) lo = mid + 1;
      else hi = mid;
    }
    const int b = lo - 1;
    const int bi = (q - s_f[b]) * bpp + i;
    if (bi >= p.max_blocks) continue;
    const int id = __ldg(p.block_tables + (size_t)b * p.max_blocks + bi);
    if (id < 0 || id >= p.num_blocks) continue;
    const size_t e = ((size_t)id * hkv + h) * BS * D;
    prefetch_l2_bulk(kc + e, kSlice);
    prefetch_l2_bulk(vc + e, kSlice);
  }
  __syncthreads();  // the scratch is the K/V ring from here on
}

// Batches (with a shared prefix) of up to this many sequences let the attention kernel
// derive the plan's first units itself.
constexpr int kEarlyMaxSeqs = 1024;

// Shared memory the attention kernel's own records take: three ints per sequence and a
// reduction scratch.
__host__ __device__ constexpr size_t early_table_bytes(int num_seqs) {
  return ((size_t)(3 * num_seqs + 64) * sizeof(int) + 15) / 16 * 16;
}

// The attention kernel's own records of the plan's first units, in a batch with a shared
// prefix.  The plan lists every sequence's full partitions (all but its last) first, in
// sequence order, and their lengths and partial slots are functions of the context
// lengths and the sharer list alone; each CTA evaluates the same functions here, into
// `tab` (early_table_bytes(num_seqs) of shared memory), so that its producers can take
// those units while the plan is still being built.  Returns the number of such units and
// sets `psz` to the partition length.  Every thread of the CTA calls it.
template <int NT>
__device__ int early_records(const DecodeParams& p, int* tab, int block_size, int& psz) {
  constexpr int kPer = kEarlyMaxSeqs / NT;
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int n = p.num_seqs;
  int* s_c = tab;          // own context length (past the prefix for a sharer)
  int* s_f = tab + n;      // index of the sequence's first full partition in the list
  int* s_r = tab + 2 * n;  // its first partial slot; bit 31: it reads the shared prefix
  long long* s_sum = reinterpret_cast<long long*>(tab + 3 * n + (n & 1));  // 8-byte aligned
  int* s_max = reinterpret_cast<int*>(s_sum + NT / 32);
  int* s_a = s_max + NT / 32;
  int* s_b = s_a + NT / 32;
  static_assert(2 * (NT / 32) + 3 * (NT / 32) + 1 <= 64, "the scratch fits the table's tail");
  // the lengths are loaded while the sharer flags are set up
  int len[kPer];
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int b = tid + k * NT;
    len[k] = b < n ? __ldcg(p.context_lens + b) : 0;
  }
  for (int b = tid; b < n; b += NT) s_r[b] = 0;
  __syncthreads();
  for (int i = tid; i < p.num_sharers; i += NT) {
    const int sb = __ldg(p.sharers + i);
    if (sb >= 0 && sb < n) s_r[sb] = 1;  // (the plan flags an index outside the batch)
  }
  __syncthreads();
  long long sum = 0;
  int mx = 0;
#pragma unroll
  for (int k = 0; k < kPer; ++k) {
    const int b = tid + k * NT;
    if (b < n) {
      const int st = s_r[b] != 0 ? p.prefix_len : 0;
      const int c = max(0, clamp_ctx(len[k], p.ctx_cap) - st);
      s_c[b] = c;
      sum += c;
      if (st > 0) mx = max(mx, c);
    }
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    sum += __shfl_xor_sync(~0u, sum, o);
    mx = max(mx, __shfl_xor_sync(~0u, mx, o));
  }
  if (lane == 0) {
    s_sum[wid] = sum;
    s_max[wid] = mx;
  }
  __syncthreads();
  long long total = 0;
  int tmax = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    total += s_sum[w];
    tmax = max(tmax, s_max[w]);
  }
  psz = batch_partition_tokens(total, tmax, p.num_kv_heads, block_size, p.forced_psz,
                               p.num_sharers, p.max_own_parts);
  // exclusive scans, in sequence order, of the partial slots (own partitions and reserved
  // prefix slots) and of the full partitions; threads own consecutive sequences
  const int per = (n + NT - 1) / NT, b0 = min(n, tid * per), b1 = min(n, b0 + per);
  int slots = 0, fulls = 0;
  for (int b = b0; b < b1; ++b) {
    const int np = (s_c[b] + psz - 1) / psz;
    slots += np + (s_r[b] != 0 ? p.prefix_splits : 0);
    fulls += np > 1 ? np - 1 : 0;
  }
  int ia = slots, ib = fulls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int ta = __shfl_up_sync(~0u, ia, o), tb = __shfl_up_sync(~0u, ib, o);
    if (lane >= o) {
      ia += ta;
      ib += tb;
    }
  }
  if (lane == 31) {
    s_a[wid] = ia;
    s_b[wid] = ib;
  }
  __syncthreads();
  int ra = ia - slots, rb = ib - fulls, ftotal = 0;
#pragma unroll
  for (int w = 0; w < NT / 32; ++w) {
    if (w < wid) {
      ra += s_a[w];
      rb += s_b[w];
    }
    ftotal += s_b[w];
  }
  for (int b = b0; b < b1; ++b) {
    const int np = (s_c[b] + psz - 1) / psz;
    const bool sh = s_r[b] != 0;
    s_f[b] = rb;
    s_r[b] = ra | (sh ? (int)0x80000000u : 0);
    ra += np + (sh ? p.prefix_splits : 0);
    rb += np > 1 ? np - 1 : 0;
  }
  __syncthreads();
  return ftotal * p.num_kv_heads;
}

// Unit u (below early_records' count) from the CTA's own records: full partition u / H_kv
// of the list for KV head u % H_kv.
__device__ __forceinline__ UnitDesc early_unit(const DecodeParams& p, const int* tab, int psz,
                                               int u) {
  const int n = p.num_seqs, hkv = p.num_kv_heads;
  const int q = u / hkv;
  int lo = 0, hi = n;  // the last sequence whose first full partition is <= q
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (tab[n + mid] <= q) lo = mid + 1;
    else hi = mid;
  }
  const int b = lo - 1;
  const int r = tab[2 * n + b];
  const bool sh = r < 0;
  const int run = r & 0x7fffffff, rs = sh ? p.prefix_splits : 0;
  const int i = q - tab[n + b];
  UnitDesc d;
  d.b = b;
  d.h = u - q * hkv;
  d.tok0 = (sh ? p.prefix_len : 0) + i * psz;
  d.ntok = psz;
  d.nparts = (tab[b] + psz - 1) / psz + rs;
  d.part_idx = run + rs + i;
  d.part_start = run;
  d.valid = 1;
  return d;
}

// Waits (bounded) for the plan's flag; returns the plan's unit count, 0 if it never came.
__device__ __forceinline__ int wait_plan_units(const DecodeParams& p) {
  const uint64_t t0 = global_timer_ns();
  int v;
  while ((v = ld_acquire_gpu(p.ws.header + 5)) == 0 && global_timer_ns() - t0 < kWaitTimeoutNs)
    __nanosleep(128);
  if (v == 0) {
    flag_status(p.status, PA_STATUS_TIMEOUT);
    return 0;
  }
  return __ldcg(p.ws.header + 1);
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(MmaCfg<D, BS, 2>::kThreads, 1)
    decode_mma_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const DecodeParams p) {
  using C = MmaCfg<D, BS, 2>;
  using M = Mma<T>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  const int G = p.group;
  const uint32_t qstride = (uint32_t)C::qstride(G);
  uint8_t* stages = base;
  uint8_t* qbuf = stages + (size_t)C::kPairs * S * C::kStageBytes;
  uint8_t* zero16 = qbuf + (size_t)C::kPairs * 2 * qstride;
  uint64_t* bars = reinterpret_cast<uint64_t*>(zero16 + 128);
  UnitDesc* descs = reinterpret_cast<UnitDesc*>(bars + C::kBars);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int pair = warp % C::kPairs;
  uint64_t* full = bars + pair * S;
  uint64_t* empty = bars + C::kPairs * S + pair * S;
  uint64_t* qfull = bars + 2 * C::kPairs * S + pair * 2;
  uint64_t* qempty = bars + 2 * C::kPairs * S + 2 * C::kPairs + pair * 2;
  UnitDesc* mydesc = descs + pair * 2;
  uint8_t* myq = qbuf + (size_t)pair * 2 * qstride;
  uint8_t* mystages = stages + (size_t)pair * S * C::kStageBytes;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kBars; ++i) mbar_init(smem_addr(bars + i), 1);
    fence_mbar_init();
  }
  if (threadIdx.x < 32) reinterpret_cast<uint32_t*>(zero16)[threadIdx.x] = 0;
  if (threadIdx.x == 32) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmv);
  }
  static_assert((size_t)C::kPairs * S * C::kStageBytes >= (2 * kPrefetchMaxSeqs + 64) * 4,
                "the prefetch scratch fits in the K/V rings");
  if (p.prefetch_bytes > 0 && p.num_seqs <= kPrefetchMaxSeqs)
    prefetch_first_units<T, D, BS, C::kThreads>(p, reinterpret_cast<int*>(stages));
  // with plan_flag set, every thread waits for the kernel launched before this one (the
  // shared prefix's) on its way out, so that this grid ends after it and the merge,
  // which waits for this grid, also waits for it
  struct WaitAtExit {
    int on;
    __device__ ~WaitAtExit() {
      if (on) griddep_wait();
    }
  } wait_at_exit{p.plan_flag};
  // with a shared prefix and `early`, the producers take the full partitions from the
  // CTA's own records and wait for the plan only when those run out
  int psz_early = 0, early_units = 0;
  const int* early_tab = reinterpret_cast<const int*>(descs + C::kPairs * 2);
  if (p.early)
    early_units = early_records<C::kThreads>(p, reinterpret_cast<int*>(descs + C::kPairs * 2), BS,
                                             psz_early);
  __shared__ int s_plan_ready;
  if (p.early) {
  } else if (p.plan_flag) {
    if (threadIdx.x == 0) {
      const uint64_t t0 = global_timer_ns();
      int v;
      while ((v = ld_acquire_gpu(p.ws.header + 5)) == 0 &&
             global_timer_ns() - t0 < kWaitTimeoutNs)
        __nanosleep(128);
      s_plan_ready = v;
      if (v == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
    }
    __syncthreads();
  } else {
    __syncthreads();
    griddep_wait();  // the plan kernel's work list is complete from here on
  }
  // (a plan that never finished leaves no work: the kernel only waits and exits; with
  // `early`, lane 0 of each producer maps the end of the plan's list to INT_MAX)
  const int total_units =
      p.early ? INT_MAX : (!p.plan_flag || s_plan_ready ? __ldcg(p.ws.header + 1) : 0);

  if (warp >= C::kPairs) {
    // ------------------------------ producer warp ------------------------------
    const uint32_t qbytes = (uint32_t)G * D * sizeof(T);
    const uint64_t policy = l2_policy_evict_first();
    uint32_t tile_it = 0, q_it = 0;
    // lane 0's claims: with `early`, first the full partitions by the early counter, then,
    // once the plan's flag is up, the rest of its list (whose counter starts past them)
    bool from_plan = !p.early;
    int plan_units = 0;
    auto claim = [&]() -> int {
      if (!from_plan) {
        const int u = atomicAdd(p.ws.header + 6, 1);
        if (u < early_units) return u;
        from_plan = true;
        plan_units = wait_plan_units(p);
      }
      const int u = atomicAdd(p.ws.header, 1);
      return p.early && u >= plan_units ? INT_MAX : u;
    };
    int next_u = 0;
    if (lane == 0) next_u = claim();
    next_u = __shfl_sync(~0u, next_u, 0);
    bool ok = true;
    while (ok) {
      const int u = next_u;
      const int qs = q_it & 1;
      if (!mbar_wait(smem_addr(qempty + qs), ((q_it >> 1) & 1) ^ 1)) { ok = false; break; }
      if (u >= total_units) {
        if (lane == 0) {
          mydesc[qs].valid = 0;
          mbar_arrive(smem_addr(qfull + qs));
        }
        griddep_launch_dependents();
        break;
      }
      UnitDesc d;
      if (u < early_units) {
        d = early_unit(p, early_tab, psz_early, u);
      } else {
        if (p.early) __syncwarp();  // lane 0 saw the plan's flag: its list is visible
        d = describe_unit(load_part(p, u), u, p.num_kv_heads);
      }
      const int ntiles = (d.ntok + BS - 1) / BS;
      // The next unit is claimed when about a ring's worth of this unit's tiles is left to
      // issue: early enough to load its record and block list while those are consumed,
      // late enough that near the end of the list no unit waits behind a busy pair while
      // others have run out.
      const int claim_at = ntiles > S ? ntiles - S : 0;
      if (ntiles == 0 && lane == 0) next_u = claim();
      const int32_t* row = p.block_tables + (size_t)d.b * p.max_blocks + d.tok0 / BS;
      int ids[kMaxPartBlocks / 32];
#pragma unroll
      for (int k = 0; k < kMaxPartBlocks / 32; ++k) {
        const int t = lane + 32 * k;
        int id = -1;
        if (t < ntiles) {
          id = __ldg(row + t);
          if (id < 0 || id >= p.num_blocks) {
            flag_status(p.status, PA_STATUS_BAD_BLOCK);
            id = -1;
          }
        }
        ids[k] = id;
      }
      if (lane == 0) {
        mydesc[qs] = d;
        const uint32_t bar = smem_addr(qfull + qs);
        mbar_arrive_expect_tx(bar, qbytes);
        bulk_load(smem_addr(myq + qs * qstride),
                  static_cast<const T*>(p.q) + ((size_t)d.b * p.num_q_heads + (size_t)d.h * G) * D,
                  qbytes, bar);
      }
      ++q_it;
      for (int t = 0; t < ntiles; ++t) {
        if (t == claim_at && lane == 0) next_u = claim();
        const int s = tile_it % S;
        if (!mbar_wait(smem_addr(empty + s), ((tile_it / S) & 1) ^ 1)) { ok = false; break; }
        const int k = t >> 5;
        int id = k == 0 ? ids[0] : k == 1 ? ids[1] : k == 2 ? ids[2] : ids[3];
        id = __shfl_sync(~0u, id, t & 31);
        if (lane == 0) {
          // a bad block id reads a box that lies wholly outside the tensor: zeros
          const int y = id < 0 ? -BS : (id * p.num_kv_heads + d.h) * BS;
          const uint32_t bar = smem_addr(full + s);
          mbar_arrive_expect_tx(bar, C::kStageBytes);
          uint8_t* st = mystages + (size_t)s * C::kStageBytes;
#pragma unroll
          for (int hb = 0; hb < C::kHalves; ++hb) {
            tma_load_2d(smem_addr(st + hb * C::kBoxBytes), &tmk, hb * 64, y, bar, policy);
            tma_load_2d(smem_addr(st + C::kTileBytes + hb * C::kBoxBytes), &tmv, hb * 64, y, bar,
                        policy);
          }
        }
        ++tile_it;
      }
      next_u = __shfl_sync(~0u, next_u, 0);
    }
    if (!ok) {
      if (lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
      // let copies already issued land before the CTA can exit
      const uint32_t first = tile_it > (uint32_t)S ? tile_it - S : 0;
      for (uint32_t i = first; i < tile_it; ++i) mbar_wait(smem_addr(full + i % S), (i / S) & 1);
    }
    return;
  }

  // ------------------------------ consumer warp ------------------------------
  constexpr int NT = BS / 8;   // 8-token score tiles per K tile
  constexpr int KS = D / 16;   // k-steps of q.K^T
  constexpr int ON = D / 8;    // 8-column output tiles
  const int g0 = lane >> 2, c4 = lane & 3;
  const bool hi_rows = G > 8;  // rows 8..15 of the padded query group are real
  const uint32_t zero_addr = smem_addr(zero16);
  if (G <= 8) {
    consume_t<T, D, BS, C>(p, mydesc, myq, qstride, qfull, qempty, full, empty, mystages,
                           zero_addr, lane);
    return;
  }
  uint32_t tile_it = 0, q_it = 0;
  for (;;) {
    const int qs = q_it & 1;
    if (!mbar_wait(smem_addr(qfull + qs), (q_it >> 1) & 1)) {
      if (lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
      return;
    }
    const UnitDesc d = mydesc[qs];
    if (!d.valid) return;

    // query group as A fragments (rows >= G read zeros)
    uint32_t qa[KS][4];
    {
      const int i = lane >> 3;
      const int r = (lane & 7) + 8 * (i & 1);
      const uint32_t rowbase = smem_addr(myq + qs * qstride) + r * (D * sizeof(T));
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        const uint32_t addr = r < G ? rowbase + (2 * kk + (i >> 1)) * 16 : zero_addr;
        ldsm_x4(addr, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_addr(qempty + qs));
    ++q_it;

    float o[ON][4];
#pragma unroll
    for (int j = 0; j < ON; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    float m0 = kNegInf, m1 = kNegInf, l0 = 0.f, l1 = 0.f;

    const int ntiles = (d.ntok + BS - 1) / BS;
    for (int t = 0; t < ntiles; ++t) {
      const int s = tile_it % S;
      if (!mbar_wait(smem_addr(full + s), (tile_it / S) & 1)) {
        if (lane == 0) flag_status(p.status, PA_STATUS_TIMEOUT);
        return;
      }
      const uint32_t kbase = smem_addr(mystages + (size_t)s * C::kStageBytes);
      const uint32_t vbase = kbase + C::kTileBytes;

      // scores: S[16 x BS] = Qpad[16 x D] . K^T
      // two accumulators per 8-token tile (even and odd k-steps): dependent chains of
      // D / 32 instead of D / 16 MMAs
      float sc[NT][4], sd[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
        sd[nt][0] = sd[nt][1] = sd[nt][2] = sd[nt][3] = 0.f;
        const int tok = nt * 8 + (lane & 7);
#pragma unroll
        for (int kk2 = 0; kk2 < D / 32; ++kk2) {
          const int cg = 4 * kk2 + (lane >> 3);
          const uint32_t addr =
              kbase + (cg >> 3) * C::kBoxBytes + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(addr, b0, b1, b2, b3);
          M::run(sc[nt], qa[2 * kk2], b0, b1);
          M::run(sd[nt], qa[2 * kk2 + 1], b2, b3);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
      }
      // scale into log2 units; tokens past the context never count
      const int limit = d.ntok - t * BS;
      float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const bool valid = nt * 8 + 2 * c4 + e < limit;
          sc[nt][e] = valid ? sc[nt][e] * p.scale_log2 : kNegInf;
          sc[nt][2 + e] = valid ? sc[nt][2 + e] * p.scale_log2 : kNegInf;
          mx0 = fmaxf(mx0, sc[nt][e]);
          mx1 = fmaxf(mx1, sc[nt][2 + e]);
        }
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(~0u, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(~0u, mx1, 2));
      const bool need0 = mx0 > m0 + kRescaleThreshold;
      const bool need1 = hi_rows && mx1 > m1 + kRescaleThreshold;
      if (__any_sync(~0u, need0 || need1)) {
        if (need0) {
          const float a = fast_exp2(m0 - mx0);
          m0 = mx0;
          l0 *= a;
#pragma unroll
          for (int j = 0; j < ON; ++j) { o[j][0] *= a; o[j][1] *= a; }
        }
        if (need1) {
          const float a = fast_exp2(m1 - mx1);
          m1 = mx1;
          l1 *= a;
#pragma unroll
          for (int j = 0; j < ON; ++j) { o[j][2] *= a; o[j][3] *= a; }
        }
      }
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        sc[nt][0] = fast_exp2(sc[nt][0] - m0);
        sc[nt][1] = fast_exp2(sc[nt][1] - m0);
        l0 += sc[nt][0] + sc[nt][1];
        if (hi_rows) {
          sc[nt][2] = fast_exp2(sc[nt][2] - m1);
          sc[nt][3] = fast_exp2(sc[nt][3] - m1);
          l1 += sc[nt][2] + sc[nt][3];
        } else {
          sc[nt][2] = sc[nt][3] = 0.f;
        }
      }
      // O[16 x D] += P[16 x BS] . V, with P carried as hi + lo 16-bit terms
#pragma unroll
      for (int ks = 0; ks < BS / 16; ++ks) {
        uint32_t ah[4], al[4];
        ah[0] = M::pack_split(sc[2 * ks][0], sc[2 * ks][1], al[0]);
        ah[1] = M::pack_split(sc[2 * ks][2], sc[2 * ks][3], al[1]);
        ah[2] = M::pack_split(sc[2 * ks + 1][0], sc[2 * ks + 1][1], al[2]);
        ah[3] = M::pack_split(sc[2 * ks + 1][2], sc[2 * ks + 1][3], al[3]);
        const int tok = 16 * ks + (lane & 7) + 8 * ((lane >> 3) & 1);
        // V rows of tokens past the context may hold anything (even NaN bits) and are
        // multiplied by P = 0: clear them in the fragments of the last tile.
        const int vlim = limit - 16 * ks;
        const bool tail = vlim < 16;
        const uint32_t m_lo0 = (2 * c4 < vlim ? 0x0000ffffu : 0u) | (2 * c4 + 1 < vlim ? 0xffff0000u : 0u);
        const uint32_t m_hi0 =
            (2 * c4 + 8 < vlim ? 0x0000ffffu : 0u) | (2 * c4 + 9 < vlim ? 0xffff0000u : 0u);
#pragma unroll
        for (int dt2 = 0; dt2 < D / 16; ++dt2) {
          const int cg = 2 * dt2 + (lane >> 4);
          const uint32_t addr =
              vbase + (cg >> 3) * C::kBoxBytes + tok * 128 + (((cg & 7) ^ (tok & 7)) << 4);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_trans(addr, b0, b1, b2, b3);
          if (tail) {
            b0 &= m_lo0;
            b1 &= m_hi0;
            b2 &= m_lo0;
            b3 &= m_hi0;
          }
          M::run(o[2 * dt2], ah, b0, b1);
          M::run(o[2 * dt2], al, b0, b1);
          M::run(o[2 * dt2 + 1], ah, b2, b3);
          M::run(o[2 * dt2 + 1], al, b2, b3);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(empty + s));
      ++tile_it;
    }

    l0 += __shfl_xor_sync(~0u, l0, 1);
    l0 += __shfl_xor_sync(~0u, l0, 2);
    l1 += __shfl_xor_sync(~0u, l1, 1);
    l1 += __shfl_xor_sync(~0u, l1, 2);
    const int hq0 = d.h * G;
    if (d.nparts == 1) {
      const size_t row0 = ((size_t)d.b * p.num_q_heads + hq0) * D;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int g = g0 + 8 * half;
        if (g >= G) continue;
        const float inv = 1.f / (half ? l1 : l0);
        const size_t at = row0 + (size_t)g * D + 2 * c4;
        if (p.out_f32) {
          float* out = static_cast<float*>(p.out) + at;
#pragma unroll
          for (int j = 0; j < ON; ++j) store2(out + j * 8, o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
        } else {
          T* out = static_cast<T*>(p.out) + at;
#pragma unroll
          for (int j = 0; j < ON; ++j) store2(out + j * 8, o[j][2 * half] * inv, o[j][2 * half + 1] * inv);
        }
      }
    } else {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const int g = g0 + 8 * half;
        if (g >= G) continue;
        const size_t slot = (size_t)d.part_idx * p.num_q_heads + hq0 + g;
        float* acc = p.ws.part_acc + slot * D + 2 * c4;
#pragma unroll
        for (int j = 0; j < ON; ++j) store2(acc + j * 8, o[j][2 * half], o[j][2 * half + 1]);
        if (c4 == 0) p.ws.part_ml[slot] = make_float2(half ? m1 : m0, half ? l1 : l0);
      }
    }
  }
}

// ----------------------------------------------------------------------------------
// 2b. attend: fp32 on CUDA cores (one warp per unit, one token at a time)
// ----------------------------------------------------------------------------------

template <int D>
__global__ void __launch_bounds__(128) decode_f32_kernel(const float* __restrict__ k_cache,
                                                         const float* __restrict__ v_cache,
                                                         const DecodeParams p, int block_size) {
  constexpr int V = D / 32;  // elements per lane
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int G = p.group;
  const int total_units = p.ws.header[1];
  for (;;) {
    int u = 0;
    if (lane == 0) u = atomicAdd(p.ws.header, 1);
    u = __shfl_sync(~0u, u, 0);
    if (u >= total_units) {
      griddep_launch_dependents();
      return;
    }
    const UnitDesc d = describe_unit(load_part(p, u), u, p.num_kv_heads);
    const float* qb = static_cast<const float*>(p.q) + ((size_t)d.b * p.num_q_heads + (size_t)d.h * G) * D;
    float qv[kMaxGroup][V], acc[kMaxGroup][V], m[kMaxGroup], l[kMaxGroup];
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      m[g] = kNegInf;
      l[g] = 0.f;
#pragma unroll
      for (int i = 0; i < V; ++i) {
        qv[g][i] = g < G ? qb[g * D + lane + 32 * i] : 0.f;
        acc[g][i] = 0.f;
      }
    }
    const int32_t* row = p.block_tables + (size_t)d.b * p.max_blocks;
    for (int tok = d.tok0; tok < d.tok0 + d.ntok; ++tok) {
      const int blk = __ldg(row + tok / block_size);
      if (blk < 0 || blk >= p.num_blocks) {
        if (lane == 0) flag_status(p.status, PA_STATUS_BAD_BLOCK);
        continue;
      }
      const size_t off = (((size_t)blk * p.num_kv_heads + d.h) * block_size + tok % block_size) * D;
      float kv[V], vv[V];
#pragma unroll
      for (int i = 0; i < V; ++i) {
        kv[i] = __ldg(k_cache + off + lane + 32 * i);
        vv[i] = __ldg(v_cache + off + lane + 32 * i);
      }
#pragma unroll
      for (int g = 0; g < kMaxGroup; ++g) {
        if (g >= G) break;
        float s = 0.f;
#pragma unroll
        for (int i = 0; i < V; ++i) s = fmaf(qv[g][i], kv[i], s);
#pragma unroll
        for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(~0u, s, o);
        const float x = s * p.scale_log2;
        const float mn = fmaxf(m[g], x);
        const float a = fast_exp2(m[g] - mn);
        const float e = fast_exp2(x - mn);
        l[g] = l[g] * a + e;
#pragma unroll
        for (int i = 0; i < V; ++i) acc[g][i] = fmaf(acc[g][i], a, e * vv[i]);
        m[g] = mn;
      }
    }
    const int hq0 = d.h * G;
#pragma unroll
    for (int g = 0; g < kMaxGroup; ++g) {
      if (g >= G) break;
      if (d.nparts == 1) {
        float* out = static_cast<float*>(p.out) + ((size_t)d.b * p.num_q_heads + hq0 + g) * D;
        const float inv = 1.f / l[g];
#pragma unroll
        for (int i = 0; i < V; ++i) out[lane + 32 * i] = acc[g][i] * inv;
      } else {
        const size_t slot = (size_t)d.part_idx * p.num_q_heads + hq0 + g;
#pragma unroll
        for (int i = 0; i < V; ++i) p.ws.part_acc[slot * D + lane + 32 * i] = acc[g][i];
        if (lane == 0) p.ws.part_ml[slot] = make_float2(m[g], l[g]);
      }
    }
  }
}

// ----------------------------------------------------------------------------------
// host side
// ----------------------------------------------------------------------------------
constexpr int kMaxDev = 64;

struct KernelSlot {
  const void* fn;
  size_t smem_max;
  int occupancy[kMaxDev];
  bool configured[kMaxDev];
};

std::mutex g_cfg_mutex;

// Sets the kernel's shared-memory limit and reads its occupancy once per device.
int configure(KernelSlot& k, int dev, int threads, size_t smem_launch) {
  std::lock_guard<std::mutex> lock(g_cfg_mutex);
  if (!k.configured[dev]) {
    if (cudaFuncSetAttribute(k.fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)k.smem_max) != cudaSuccess)
      return -1;
    int occ = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k.fn, threads, k.smem_max) !=
        cudaSuccess)
      return -1;
    k.occupancy[dev] = occ < 1 ? 1 : occ;
    k.configured[dev] = true;
  }
  (void)smem_launch;
  return k.occupancy[dev];
}

template <typename T, int D, int BS>
KernelSlot& mma_slot() {
  static KernelSlot slot = {reinterpret_cast<const void*>(&decode_mma_kernel<T, D, BS>),
                            MmaCfg<D, BS, 2>::smem_bytes(kMaxGroup), {}, {}};
  return slot;
}

template <typename T, int D, int BS>
int launch_mma(const DecodeArgs& a, const DecodeParams& p, cudaStream_t stream) {
  using C = MmaCfg<D, BS, 2>;
  CUtensorMap tmk, tmv;
  int r1 = encode_cache_map(&tmk, a.k_cache, a.dtype, a.num_blocks, a.num_kv_heads, a.block_size,
                            a.head_dim);
  int r2 = encode_cache_map(&tmv, a.v_cache, a.dtype, a.num_blocks, a.num_kv_heads, a.block_size,
                            a.head_dim);
  if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS)
    return fail(PA_ERR_CUDA, "pa_decode: cuTensorMapEncodeTiled failed (%d, %d)", r1, r2);
  int dev = 0;
  cudaGetDevice(&dev);
  KernelSlot& slot = mma_slot<T, D, BS>();
  const int occ = configure(slot, dev, C::kThreads, slot.smem_max);
  if (occ < 0) return fail(PA_ERR_CUDA, "pa_decode: kernel configuration failed");
  const int grid = a.max_ctas > 0 ? std::min(a.max_ctas, sm_count() * occ) : sm_count() * occ;
  const size_t smem = C::smem_bytes(p.group) + (p.early ? early_table_bytes(p.num_seqs) : 0);
  const cudaError_t e = launch_pdl(decode_mma_kernel<T, D, BS>, dim3(grid), dim3(C::kThreads),
                                   smem, stream, tmk, tmv, p);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode: %s", cudaGetErrorString(e));
  return PA_OK;
}

// Whether the attention kernel's own records of the plan's first units fit beside its
// rings (within the shared memory its launches are configured for).
bool early_table_fits(int head_dim, int block_size, int group, int num_seqs) {
  auto fits = [&](size_t base, size_t limit) {
    return base + early_table_bytes(num_seqs) <= limit;
  };
  if (head_dim == 128 && block_size == 16)
    return fits(MmaCfg<128, 16, 2>::smem_bytes(group), MmaCfg<128, 16, 2>::smem_bytes(kMaxGroup));
  if (head_dim == 128 && block_size == 32)
    return fits(MmaCfg<128, 32, 2>::smem_bytes(group), MmaCfg<128, 32, 2>::smem_bytes(kMaxGroup));
  if (head_dim == 64 && block_size == 16)
    return fits(MmaCfg<64, 16, 2>::smem_bytes(group), MmaCfg<64, 16, 2>::smem_bytes(kMaxGroup));
  if (head_dim == 64 && block_size == 32)
    return fits(MmaCfg<64, 32, 2>::smem_bytes(group), MmaCfg<64, 32, 2>::smem_bytes(kMaxGroup));
  return false;
}

template <typename T>
int launch_mma_dispatch(const DecodeArgs& a, const DecodeParams& p, cudaStream_t stream) {
  if (a.head_dim == 128 && a.block_size == 16) return launch_mma<T, 128, 16>(a, p, stream);
  if (a.head_dim == 128 && a.block_size == 32) return launch_mma<T, 128, 32>(a, p, stream);
  if (a.head_dim == 64 && a.block_size == 16) return launch_mma<T, 64, 16>(a, p, stream);
  if (a.head_dim == 64 && a.block_size == 32) return launch_mma<T, 64, 32>(a, p, stream);
  return fail(PA_ERR_UNSUPPORTED, "pa_decode: head_dim %d / block_size %d", a.head_dim,
              a.block_size);
}

}  // namespace

size_t decode_max_parts(int num_seqs, int num_kv_heads, int max_ctx, int block_size,
                        int forced_psz) {
  if (forced_psz > 0)
    return (size_t)((long long)num_seqs * (((long long)max_ctx + forced_psz - 1) / forced_psz) +
                    num_seqs);
  const long long pmax = (long long)kMaxPartBlocks * block_size;
  const long long by_target = (kTargetUnits + num_kv_heads - 1) / num_kv_heads;
  const long long by_length = (long long)num_seqs * ((max_ctx + pmax - 1) / pmax);
  return (size_t)(std::max(by_target, by_length) + num_seqs);
}

namespace {
struct WsLayout {
  size_t header, part_start, seq_flags, merge_seqs, units, part_ml, part_acc, total;
};
WsLayout decode_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int max_ctx,
                       int block_size, long long extra_slots, int forced_psz) {
  const size_t parts = decode_max_parts(num_seqs, num_kv_heads, max_ctx, block_size, forced_psz);
  const size_t slots = parts + (size_t)extra_slots;
  WsLayout l;
  l.header = 0;
  l.part_start = 256;
  l.seq_flags = align_up(l.part_start + sizeof(int) * (num_seqs + 1), 256);
  l.merge_seqs = align_up(l.seq_flags + (extra_slots > 0 ? sizeof(int) * num_seqs : 0), 256);
  l.units = align_up(l.merge_seqs + sizeof(int) * num_seqs, 256);
  l.part_ml = align_up(l.units + sizeof(PartRec) * parts, 256);
  l.part_acc = align_up(l.part_ml + sizeof(float2) * slots * num_q_heads, 256);
  l.total = align_up(l.part_acc + sizeof(float) * slots * num_q_heads * head_dim, 256);
  return l;
}
}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                              int max_ctx, int block_size, long long extra_slots,
                              int forced_psz) {
  return decode_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx, block_size,
                       extra_slots, forced_psz)
      .total;
}

DecodeWorkspace carve_decode_workspace(void* ws, int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int max_ctx, int block_size,
                                       long long extra_slots, int forced_psz) {
  const WsLayout l = decode_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, max_ctx,
                                   block_size, extra_slots, forced_psz);
  uint8_t* b = static_cast<uint8_t*>(ws);
  DecodeWorkspace w;
  w.header = reinterpret_cast<int*>(b + l.header);
  w.part_start = reinterpret_cast<int*>(b + l.part_start);
  w.seq_flags = extra_slots > 0 ? reinterpret_cast<int*>(b + l.seq_flags) : nullptr;
  w.merge_seqs = reinterpret_cast<int*>(b + l.merge_seqs);
  w.parts = reinterpret_cast<PartRec*>(b + l.units);
  w.part_ml = reinterpret_cast<float2*>(b + l.part_ml);
  w.part_acc = reinterpret_cast<float*>(b + l.part_acc);
  return w;
}

PrefixPlan plan_prefix(int num_sharers, int prefix_len, int group, int num_kv_heads) {
  PrefixPlan pp = {};
  pp.num_sharers = num_sharers;
  pp.prefix_len = prefix_len;
  if (num_sharers <= 0 || prefix_len <= 0) {
    pp.num_sharers = 0;
    pp.splits = 0;
    return pp;
  }
  // about 64 CTAs (42% of 152 SMs): the attention over the sequences' own contexts takes
  // the other SMs meanwhile (a constant, so that the workspace size does not depend on
  // the device)
  constexpr int kTile = 128, kRowsPerCta = 256, kTargetCtas = 64;
  const long long row_ctas = ((long long)num_sharers * group + kRowsPerCta - 1) / kRowsPerCta;
  const long long tiles = (prefix_len + kTile - 1) / kTile;
  long long want = (kTargetCtas + row_ctas * num_kv_heads - 1) / (row_ctas * num_kv_heads);
  want = std::max(1ll, std::min(want, tiles));
  const long long split_tiles = (tiles + want - 1) / want;
  pp.split_tokens = (int)(split_tiles * kTile);
  pp.splits = (int)((prefix_len + pp.split_tokens - 1) / pp.split_tokens);
  return pp;
}

int launch_decode(const DecodeArgs& a, cudaStream_t stream) {
  if (a.num_seqs > 65535) return fail(PA_ERR_UNSUPPORTED, "pa_decode: more than 65535 sequences");
  const long long cap = std::min<long long>(a.max_ctx, (long long)a.max_blocks * a.block_size);
  const int ctx_cap = (int)std::min<long long>(cap, 0x7fffffffll);
  const int out_row_vec16 =
      (int)((size_t)a.num_q_heads * a.head_dim * dtype_bytes(a.out_dtype) / 16);

  // one CTA; a thread per sequence up to 1,024 threads (fewer warps meet in its barriers)
  const int plan_threads = std::min(1024, std::max(32, (a.num_seqs + 31) / 32 * 32));
  PrefixPlan pre = a.prefix;
  pre.max_own_parts = merge_one_round(a.head_dim) - pre.splits;
  // With a shared prefix the attention kernel may take the plan's first units from its
  // own records (not when the plan waits for the kernel before it only at its end: the
  // attention kernel would then start before that kernel is done)
  const bool early = a.prefix.num_sharers > 0 && !a.plan_wait_late && a.dtype != PA_F32 &&
                     a.num_seqs <= kEarlyMaxSeqs &&
                     early_table_fits(a.head_dim, a.block_size, a.num_q_heads / a.num_kv_heads,
                                      a.num_seqs);
  cudaError_t e = launch_pdl(decode_plan_kernel, dim3(1), dim3(plan_threads), 0, stream, a.context_lens,
                             a.num_seqs, ctx_cap, a.num_kv_heads, a.block_size, a.ws, a.status,
                             static_cast<int4*>(a.out), out_row_vec16, pre,
                             a.plan_wait_late ? 1 : 0, a.forced_part_tokens, early ? 1 : 0);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode (plan): %s", cudaGetErrorString(e));
  if (a.prefix.num_sharers > 0) {
    const int rc = launch_shared_prefix(a, stream);
    if (rc != PA_OK) return rc;
  }
  DecodeParams p;
  p.q = a.q;
  p.out = a.out;
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.ws = a.ws;
  p.status = a.status;
  p.max_blocks = a.max_blocks;
  p.ctx_cap = ctx_cap;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.out_f32 = a.out_dtype == PA_F32 && a.dtype != PA_F32;
  p.out_bytes = (int)dtype_bytes(a.out_dtype);
  p.out_bf16 = a.out_dtype == PA_BF16;
  p.scale_log2 = a.scale * kLog2e;
  p.k_cache = a.k_cache;
  p.v_cache = a.v_cache;
  // the first partitions' K/V that HBM can bring in while the plan is built (not with a
  // shared prefix, whose sequences' partitions start after it)
  p.prefetch_bytes = a.prefix.num_sharers > 0 ? 0 : kDecodePrefetchBytes;
  p.plan_flag = a.prefix.num_sharers > 0;
  p.forced_psz = a.forced_part_tokens;
  p.sharers = pre.sharers;
  p.num_sharers = pre.num_sharers;
  p.prefix_len = pre.prefix_len;
  p.prefix_splits = pre.splits;
  p.max_own_parts = pre.max_own_parts;
  p.early = early ? 1 : 0;

  int rc = PA_OK;
  if (a.dtype == PA_F32) {
    const int ctas = std::max(1, sm_count()) * 8;
    const dim3 grid(a.max_ctas > 0 ? std::min(ctas, a.max_ctas * 8) : ctas);
    const float* kc = static_cast<const float*>(a.k_cache);
    const float* vc = static_cast<const float*>(a.v_cache);
    e = a.head_dim == 128
            ? launch_pdl(decode_f32_kernel<128>, grid, dim3(128), 0, stream, kc, vc, p, a.block_size)
            : launch_pdl(decode_f32_kernel<64>, grid, dim3(128), 0, stream, kc, vc, p, a.block_size);
    if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode: %s", cudaGetErrorString(e));
  } else if (a.dtype == PA_BF16) {
    rc = launch_mma_dispatch<__nv_bfloat16>(a, p, stream);
  } else {
    rc = launch_mma_dispatch<__half>(a, p, stream);
  }
  if (rc != PA_OK) return rc;
  // rows to merge are known only on the device: at most every (sequence, query head),
  // in a grid of up to kMergeCtasPerSm CTAs per SM
  const long long warps = (long long)a.num_seqs * a.num_q_heads;
  const int merge_ctas = (int)std::min<long long>((warps + 7) / 8,
                                                  (long long)sm_count() * kMergeCtasPerSm);
  const MergeKernel merge =
      a.head_dim == 128 ? merge_kernel_for<128>(a.out_dtype) : merge_kernel_for<64>(a.out_dtype);
  e = launch_pdl(merge, dim3(std::max(1, merge_ctas)), dim3(256), 0, stream, p);
  if (e != cudaSuccess) return fail(PA_ERR_CUDA, "pa_decode (merge): %s", cudaGetErrorString(e));
  return PA_OK;
}

}  // namespace pa
