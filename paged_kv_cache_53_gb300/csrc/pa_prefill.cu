// Chunked-prefill attention over paged context on sm_103a tensor cores (tcgen05).
//
// A chunk of prompt tokens attends causally to its sequence's whole context, the chunk
// included ("PagedAttention and Continuous Batching Explained (2026)", section "Chunked
// prefill").  The work is a dense contraction: for KV head h, the (chunk token, query
// head of h's group) pairs form the rows of Q, and each 64-token tile of context is a
// K/V block of the product.
//
// One CTA owns 128 query rows of one (sequence, KV head); row r is token r / G of its
// slice of the chunk and query head h * G + r % G, so a tile covers 128 / G consecutive
// chunk tokens and every row of it shares the same K/V.  Warp roles:
//   warp 0     TMA producer: the Q tile once (a 3-D box over [token, head, dim]), then
//              every K/V tile (one 2-D box per block and 64-column half, gathered
//              through the block table, 128-byte swizzle) into a 3-stage ring.
//   warp 1     MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM buffers, then
//              O += P_j V_j into a TMEM accumulator, with P_j carried as the sum of a
//              bf16/fp16 "hi" term and the rounding residual "lo" (two MMAs), since a
//              single 16-bit P alone can miss a 2e-3 absolute tolerance on short
//              contexts.  tcgen05.commit signals the barriers.
//   warps 4-7  softmax, one thread per row: read S_j from TMEM, apply scale and the
//              causal mask, keep the running max (moved only when it grows by more than
//              2^8, rescaling O in TMEM then) and sum, write P_j to swizzled shared
//              memory; at the end normalise O and store the rows.
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

struct PrefillParams {
  void* out;
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* context_lens;
  int32_t* status;
  int max_blocks, num_q_heads, num_kv_heads, group, num_blocks, out_f32;
  float scale_log2;
};

template <int D, int BS>
struct PrefillCfg {
  static constexpr int BM = 128;                       // query rows per CTA
  static constexpr int BN = 64;                        // context tokens per K/V tile
  static constexpr int kHalves = D / 64;               // 128-byte column groups
  static constexpr int kQHalfBytes = BM * 128;         // 16 KiB
  static constexpr int kQBytes = kHalves * kQHalfBytes;
  static constexpr int kKvHalfBytes = BN * 128;        // 8 KiB
  static constexpr int kKBytes = kHalves * kKvHalfBytes;
  static constexpr int kStageBytes = 2 * kKBytes;      // K then V
  static constexpr int kStages = 3;
  static constexpr int kPBytes = BM * BN * 2;          // one 16-bit P term, 16 KiB
  static constexpr int kPBufBytes = 2 * kPBytes;       // hi + lo
  static constexpr int kBlocksPerTile = BN / BS;
  static constexpr int kThreads = 256;
  static constexpr int kTmemCols = 256;                // S0 | S1 | O
  // barriers: q_full, kv_full[3], kv_empty[3], s_full[2], s_free[2], p_full[2],
  // p_empty[2], o_full
  static constexpr int kBars = 16;
  static constexpr size_t kSmem =
      1024 + kQBytes + (size_t)kStages * kStageBytes + 2 * kPBufBytes + kBars * 8 + 16;
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

// Packs 8 floats into 16-bit hi terms and their rounding residuals.
template <typename T>
__device__ __forceinline__ void pack8_split(const float* v, uint4& hi, uint4& lo) {
  uint32_t h[4], l[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = Mma<T>::pack_split(v[2 * i], v[2 * i + 1], l[i]);
  hi = make_uint4(h[0], h[1], h[2], h[3]);
  lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

template <typename T, int D, int BS>
__global__ void __launch_bounds__(256, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmq, const __grid_constant__ CUtensorMap tmk,
                   const __grid_constant__ CUtensorMap tmv, const PrefillParams p) {
  using C = PrefillCfg<D, BS>;
  constexpr int BN = C::BN, S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~uintptr_t(1023));
  uint8_t* sQ = base;
  uint8_t* sKV = sQ + C::kQBytes;
  uint8_t* sP = sKV + S * C::kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(sP + 2 * C::kPBufBytes);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + C::kBars);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = bars + 1 + S;
  uint64_t* s_full = bars + 1 + 2 * S;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;
  uint64_t* p_empty = p_full + 2;
  uint64_t* o_full = p_empty + 2;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qtile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int G = p.group;
  const int tpt = C::BM / G;  // chunk tokens per tile

  griddep_wait();  // the chunk's K/V were written by the preceding cache write
  const int q_begin = __ldg(p.cu_q_lens + b);
  const int chunk = __ldg(p.cu_q_lens + b + 1) - q_begin;
  const int t0 = qtile * tpt;
  if (t0 >= chunk) return;  // the whole CTA leaves before touching any barrier
  const int ctx = __ldg(p.context_lens + b);
  if (ctx < chunk || (long long)ctx > (long long)p.max_blocks * BS) {
    if (threadIdx.x == 0 && qtile == 0) flag_status(p.status, PA_STATUS_BAD_CONTEXT);
    return;
  }
  const int ctx0 = ctx - chunk;
  const int ntok = min(tpt, chunk - t0);    // chunk tokens of this tile
  const int rows_valid = ntok * G;
  const int last_pos = ctx0 + t0 + ntok - 1;  // position of the tile's last query
  const int n_kv = last_pos / BN + 1;         // K/V tiles it needs
  const int nblk_ctx = (ctx + BS - 1) / BS;

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(q_full), 1);
    for (int i = 0; i < S; ++i) {
      mbar_init(smem_addr(kv_full + i), 1);
      mbar_init(smem_addr(kv_empty + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_addr(s_full + i), 1);
      mbar_init(smem_addr(s_free + i), 128);
      mbar_init(smem_addr(p_full + i), 128);
      mbar_init(smem_addr(p_empty + i), 1);
    }
    mbar_init(smem_addr(o_full), 1);
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
  bool ok = true;

  if (warp == 0) {
    // ------------------------------ TMA producer ------------------------------
    const uint64_t keep = l2_policy_evict_last();  // K/V tiles are re-read by other tiles
    if (lane == 0) {
      mbar_arrive_expect_tx(smem_addr(q_full), C::kQBytes);
#pragma unroll
      for (int hb = 0; hb < C::kHalves; ++hb)
        tma_load_3d(smem_addr(sQ + hb * C::kQHalfBytes), &tmq, hb * 64, h * G, q_begin + t0,
                    smem_addr(q_full), keep);
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
    if (lane == 0) {
      const uint32_t id_s = tc::idesc_f16(Fmt<T>::v, C::BM, BN, false, false);
      const uint32_t id_o = tc::idesc_f16(Fmt<T>::v, C::BM, D, false, true);
      const uint32_t tO = tmem + 2 * BN;
      auto issue_pv = [&](int jj) -> bool {
        if (!mbar_wait(smem_addr(p_full + (jj & 1)), (jj >> 1) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t sv = smem_addr(sKV + (jj % S) * C::kStageBytes + C::kKBytes);
        const uint32_t sp = smem_addr(sP + (jj & 1) * C::kPBufBytes);
#pragma unroll
        for (int ks = 0; ks < BN / 16; ++ks) {
          const uint64_t bdesc = tc::smem_desc_sw128(sv + ks * 16 * 128, C::kKvHalfBytes, 1024);
          const uint64_t ahi = tc::smem_desc_sw128(sp + ks * 32, 16, 1024);
          const uint64_t alo = tc::smem_desc_sw128(sp + C::kPBytes + ks * 32, 16, 1024);
          tc::mma_f16_ss(tO, ahi, bdesc, id_o, jj > 0 || ks > 0);
          tc::mma_f16_ss(tO, alo, bdesc, id_o, true);
        }
        tc::commit(smem_addr(p_empty + (jj & 1)));
        tc::commit(smem_addr(kv_empty + (jj % S)));
        return true;
      };
      if (!mbar_wait(smem_addr(q_full), 0)) ok = false;
      for (int j = 0; j < n_kv && ok; ++j) {
        const int s = j % S;
        if (!mbar_wait(smem_addr(kv_full + s), (j / S) & 1)) { ok = false; break; }
        if (j >= 2 && !mbar_wait(smem_addr(s_free + (j & 1)), ((j - 2) >> 1) & 1)) { ok = false; break; }
        tc::fence_after_sync();
        const uint32_t tS = tmem + (j & 1) * BN;
        const uint32_t sq = smem_addr(sQ), sk = smem_addr(sKV + s * C::kStageBytes);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t koff = (kk & 3) * 32;
          const uint64_t a = tc::smem_desc_sw128(sq + (kk >> 2) * C::kQHalfBytes + koff, 16, 1024);
          const uint64_t bd = tc::smem_desc_sw128(sk + (kk >> 2) * C::kKvHalfBytes + koff, 16, 1024);
          tc::mma_f16_ss(tS, a, bd, id_s, kk > 0);
        }
        tc::commit(smem_addr(s_full + (j & 1)));
        if (j >= 1 && !issue_pv(j - 1)) { ok = false; break; }
      }
      if (ok && !issue_pv(n_kv - 1)) ok = false;
      if (ok) tc::commit(smem_addr(o_full));
      if (!ok) flag_status(p.status, PA_STATUS_TIMEOUT);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------ softmax / epilogue ------------------------------
    const int r = threadIdx.x - 128;                         // row of the tile = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int rpos = ctx0 + t0 + r / G;                      // position of this row's query
    float m = kNegInf, l = 0.f;
    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait(smem_addr(s_full + (j & 1)), (j >> 1) & 1)) { ok = false; break; }
      tc::fence_after_sync();
      float x[BN];
      tc::tmem_ld32(trow + (j & 1) * BN, *reinterpret_cast<float(*)[32]>(x));
      tc::tmem_ld32(trow + (j & 1) * BN + 32, *reinterpret_cast<float(*)[32]>(x + 32));
      tc::tmem_wait_ld();
      tc::fence_before_sync();
      mbar_arrive(smem_addr(s_free + (j & 1)));

      const int kp0 = j * BN;
      float mx = kNegInf;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        x[c] = (kp0 + c <= rpos) ? x[c] * p.scale_log2 : kNegInf;
        mx = fmaxf(mx, x[c]);
      }
      const bool need = mx > m + kRescaleThreshold;
      if (__any_sync(~0u, need)) {
        const float alpha = need ? fast_exp2(m - mx) : 1.f;
        if (j > 0) {
          // O holds P_0..j-1 V: wait for the last of those products, then rescale
          if (!mbar_wait(smem_addr(p_empty + ((j - 1) & 1)), ((j - 1) >> 1) & 1)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll
          for (int c0 = 0; c0 < D; c0 += 32) {
            float o[32];
            tc::tmem_ld32(trow + 2 * BN + c0, o);
            tc::tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tc::tmem_st32(trow + 2 * BN + c0, o);
          }
          tc::tmem_wait_st();
        }
        if (need) {
          l *= alpha;
          m = mx;
        }
      }
      float sum = 0.f;
#pragma unroll
      for (int c = 0; c < BN; ++c) {
        x[c] = fast_exp2(x[c] - m);
        sum += x[c];
      }
      l += sum;
      if (j >= 2 && !mbar_wait(smem_addr(p_empty + (j & 1)), ((j - 2) >> 1) & 1)) { ok = false; break; }
      const uint32_t sp = smem_addr(sP + (j & 1) * C::kPBufBytes) + r * 128;
#pragma unroll
      for (int c8 = 0; c8 < BN / 8; ++c8) {
        uint4 hi, lo;
        pack8_split<T>(x + 8 * c8, hi, lo);
        const uint32_t off = (uint32_t)((c8 ^ (r & 7)) << 4);
        st_shared_v4(sp + off, hi);
        st_shared_v4(sp + C::kPBytes + off, lo);
      }
      if (j == n_kv - 1) {
        // V rows of the last tile past the context (inside its last block) may hold
        // anything, NaN bits included, and would meet P = 0: zero them
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
        }
      }
      tc::fence_proxy_async_smem();
      tc::fence_before_sync();
      mbar_arrive(smem_addr(p_full + (j & 1)));
    }
    // epilogue: O / l -> out rows
    if (ok && mbar_wait(smem_addr(o_full), 0)) {
      tc::fence_after_sync();
      const float inv = 1.f / l;
      const size_t orow = ((size_t)(q_begin + t0 + r / G) * p.num_q_heads + h * G + r % G) * D;
#pragma unroll
      for (int c0 = 0; c0 < D; c0 += 32) {
        float o[32];
        tc::tmem_ld32(trow + 2 * BN + c0, o);
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
  const long long tiles = ((long long)a.max_q * G + C::BM - 1) / C::BM;
  if (tiles > 0x7fffffffll || a.num_seqs > 65535 || a.num_kv_heads > 65535)
    return fail(PA_ERR_UNSUPPORTED, "pa_prefill_chunk: grid too large");
  const cudaError_t e = launch_pdl(prefill_kernel<T, D, BS>,
                                   dim3((unsigned)tiles, a.num_kv_heads, a.num_seqs),
                                   dim3(C::kThreads), C::kSmem, stream, tmq, tmk, tmv, p);
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

size_t prefill_workspace_bytes(int, int, int, int, int, int, int, int) { return 0; }

int launch_prefill(const PrefillArgs& a, cudaStream_t stream) {
  return a.dtype == PA_BF16 ? dispatch<__nv_bfloat16>(a, stream) : dispatch<__half>(a, stream);
}

}  // namespace pa
