// Absorb BMMs either side of the latent decode ("[ROCm] Dspark MLA module",
// Details: the decode's absorb BMM, FP8/FP4 BMM when enabled, else torch.bmm):
//   before: q_lat[t, h, :] = q_nope[t, h, :] @ W_UK[h]     (k = 128, n = 512)
//   after:  out[t, h, :]   = o_lat[t, h, :]  @ W_UV[h]     (k = 512, n = 128)
// One kernel computes y[t, h, j] = bf16(s * sum_k x[t, h, k] * w[h, k, j]).
//
// A decode step has few tokens and many heads, so the product is computed
// transposed, D[j, t] = sum_k w[h, k, j] * x[t, h, k], with the weight as the
// M = 128 operand and the tokens as the N operand (16..256 wide): one CTA per
// (head, 128 weight columns, token tile), no padding of a small token count to
// 128 rows.  Per 64-wide k chunk, TMA brings
//   * the weight tile, [64 k][128 j]: bf16 as two 128-byte-swizzled boxes of 64 j
//     (the MN-major A operand of tcgen05.mma), fp8 as one raw 128-byte box that four
//     conversion warps expand exactly to bf16 in that same layout;
//   * the token tile, [tok_tile t][64 k] bf16, 128-byte swizzled (the K-major B
//     operand); rows past the last token are zero-filled by the TMA.
// Four MMAs (K = 16 each) per chunk accumulate D[128, tok_tile] fp32 in TMEM.  The
// epilogue warps read their 32 TMEM lanes (32 output columns j), scale, round to
// bf16 and transpose through 2 KB of shared memory per warp so each token's 32
// columns leave as one 64-byte segment.
//
// Warp roles (192 threads): 0 TMA producer, 1 TMEM allocation + MMA issue, 2-5
// fp8 conversion during the main loop and the epilogue after it.  Every barrier
// wait is bounded; a wait that runs out records MLA_DEV_WAIT_TIMEOUT (and the
// wait site) in the optional status word, raises an abort flag, and the CTA
// drains its copies and MMAs in flight (again bounded) before it frees TMEM and
// returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "tc_primitives.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kThreads = 192;
constexpr int kKChunk = 64;                    // k per pipeline stage
constexpr int kWTileBytes = 128 * kKChunk * 2;  // bf16 weight tile [64 k][128 j]
constexpr int kWBlockBytes = kWTileBytes / 2;   // one 64-column block of it
constexpr int kWRawBytes = 128 * kKChunk;       // fp8 weight tile
constexpr int kMaxStages = 4;
constexpr int kSmemAlign = 1024;

struct BmmParams {
  __nv_bfloat16* out;
  long long o_ts, o_hs;  // elements
  float w_scale;
  int n_tok, H, K, N;
  int tok_tile;          // multiple of 16, 16..256
  int stages;            // 1..kMaxStages
  int n_mtiles;          // N / 128
  int tmem_cols;         // power of two >= max(32, tok_tile)
  int stage_bytes;       // bf16 weight tile + token tile (+ raw fp8 tile)
  int32_t* status;       // optional
};

struct BmmBars {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t conv[kMaxStages];
  uint64_t acc_full;
  uint64_t drain;
  uint32_t tmem_slot;
  int abort;
};

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, int32_t c0, int32_t c1, int32_t c2,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tmap), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

// Two e4m3fn codes (low byte first) -> two bf16 values, exactly: e4m3 -> f16 is
// exact, f16 -> f32 is exact, and every e4m3 value is a bf16 value.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(two));
  float lo, hi;
  asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(h2));
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void record_timeout(const BmmParams& p, volatile int* abort, int site) {
  if (p.status && atomicCAS(p.status, 0, (int32_t)MLA_DEV_WAIT_TIMEOUT) == 0) p.status[1] = site;
  *abort = 1;
}

template <bool kFp8>
__global__ void __launch_bounds__(kThreads, 1)
    mla_absorb_bmm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                          const BmmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + kSmemAlign - 1) & ~(uintptr_t)(kSmemAlign - 1));
  BmmBars* bars = reinterpret_cast<BmmBars*>(smem + p.stages * p.stage_bytes);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mtile = blockIdx.x % p.n_mtiles, ttile = blockIdx.x / p.n_mtiles;
  const int h = blockIdx.y;
  const int m0 = mtile * 128, t0 = ttile * p.tok_tile;
  const int nk = p.K / kKChunk;
  const int x_bytes = p.tok_tile * 128;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->conv[s], 128);
    }
    mbar_init(&bars->acc_full, 1);
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_x);
    prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, (uint32_t)p.tmem_cols);
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      for (int c = 0; c < nk; ++c) {
        const int s = c % p.stages;
        if (!mbar_wait(&bars->empty[s], ((c / p.stages) & 1) ^ 1, abort)) {
          if (!*abort) record_timeout(p, abort, 1);
          break;
        }
        const uint32_t st = sbase + (uint32_t)(s * p.stage_bytes);
        mbar_arrive_expect_tx(&bars->full[s], (uint32_t)(x_bytes + (kFp8 ? kWRawBytes : kWTileBytes)));
        tma_load_3d(st + kWTileBytes, &tmap_x, c * kKChunk, h, t0, &bars->full[s]);
        if (kFp8) {
          tma_load_3d(st + kWTileBytes + x_bytes, &tmap_w, m0, c * kKChunk, h, &bars->full[s]);
        } else {
          tma_load_3d(st, &tmap_w, m0, c * kKChunk, h, &bars->full[s]);
          tma_load_3d(st + kWBlockBytes, &tmap_w, m0 + 64, c * kKChunk, h, &bars->full[s]);
        }
        ++issued;
      }
      if (*abort) {
        // Let the copies already issued land before the shared memory goes away.
        for (int c = issued > p.stages ? issued - p.stages : 0; c < issued; ++c) {
          const int s = c % p.stages;
          const long long t0c = clock64();
          while (!mbar_try_wait(&bars->full[s], (c / p.stages) & 1) && clock64() - t0c < kWaitLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, p.tok_tile, true, false);
      int issued = 0;
      for (int c = 0; c < nk; ++c) {
        const int s = c % p.stages;
        const uint32_t ph = (c / p.stages) & 1;
        if (!mbar_wait(kFp8 ? &bars->conv[s] : &bars->full[s], ph, abort)) {
          if (!*abort) record_timeout(p, abort, 2);
          break;
        }
        fence_after_sync();
        const uint32_t st = sbase + (uint32_t)(s * p.stage_bytes);
        const uint64_t adesc = smem_desc_sw128(st, kWBlockBytes, 1024);
        const uint64_t bdesc = smem_desc_sw128(st + kWTileBytes, 16, 1024);
#pragma unroll
        for (int k = 0; k < kKChunk / 16; ++k)
          mma_ss(tmem, adesc + (uint64_t)((k * 2048) >> 4), bdesc + (uint64_t)((k * 32) >> 4), idesc,
                 (c > 0 || k > 0) ? 1u : 0u);
        mma_commit(&bars->empty[s]);
        ++issued;
      }
      if (*abort) {
        if (issued > 0) {
          mma_commit(&bars->drain);
          const long long t0c = clock64();
          while (!mbar_try_wait(&bars->drain, 0) && clock64() - t0c < kWaitLimitCycles) {
          }
        }
      } else {
        mma_commit(&bars->acc_full);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ warps 2-5
    const int tid = threadIdx.x - 64;  // 0..127
    bool ok = true;
    if (kFp8) {
      for (int c = 0; c < nk && ok; ++c) {
        const int s = c % p.stages;
        if (!mbar_wait(&bars->full[s], (c / p.stages) & 1, abort)) {
          if (!*abort) record_timeout(p, abort, 3);
          ok = false;
          break;
        }
        uint8_t* st = smem + s * p.stage_bytes;
        const uint8_t* raw = st + kWTileBytes + x_bytes;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int u = tid + 128 * i;          // 16-byte unit of the raw tile: 64 rows x 8
          const int kr = u >> 3, col = (u & 7) * 16;
          const uint4 v = *reinterpret_cast<const uint4*>(raw + kr * 128 + col);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            o[2 * q] = e4m3x2_to_bf16x2((uint16_t)(w4[q] & 0xFFFFu));
            o[2 * q + 1] = e4m3x2_to_bf16x2((uint16_t)(w4[q] >> 16));
          }
          const int blk = col >> 6, uu = (col & 63) >> 3;  // 64-column block, 16-byte unit in its line
          uint8_t* line = st + blk * kWBlockBytes + kr * 128;
          *reinterpret_cast<uint4*>(line + ((uu ^ (kr & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(line + (((uu + 1) ^ (kr & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        mbar_arrive(&bars->conv[s]);
      }
    }
    if (ok && mbar_wait(&bars->acc_full, 0, abort)) {
      fence_after_sync();
      const int quad = warp & 3;                      // TMEM lanes 32*quad .. +31
      uint8_t* stg = smem + (warp - 2) * 2048;        // stage memory is free once D is complete
      __nv_bfloat16* stg_h = reinterpret_cast<__nv_bfloat16*>(stg);
      const int jcol = m0 + 32 * quad;
      for (int j0 = 0; j0 < p.tok_tile; j0 += 32) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * quad) << 16) + (uint32_t)j0, r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 32; ++i)
          stg_h[i * 32 + lane] = __float2bfloat16_rn(__uint_as_float(r[i]) * p.w_scale);
        __syncwarp();
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
          const int ti = pass * 8 + (lane >> 2);
          const int t = t0 + j0 + ti;
          if (j0 + ti < p.tok_tile && t < p.n_tok) {
            const uint4 v = *reinterpret_cast<const uint4*>(stg + ti * 64 + (lane & 3) * 16);
            *reinterpret_cast<uint4*>(p.out + (long long)t * p.o_ts + (long long)h * p.o_hs + jcol +
                                      (lane & 3) * 8) = v;
          }
        }
        __syncwarp();
      }
    } else if (ok && !*abort) {
      record_timeout(p, abort, 4);
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, (uint32_t)p.tmem_cols);
}

// ----------------------------------------------------------------------- host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return nullptr;
    fn = reinterpret_cast<EncodeTiledFn>(f);
  }
  return fn;
}

int pow2_at_least(int v) {
  int r = 1;
  while (r < v) r <<= 1;
  return r;
}

}  // namespace

mla_status launch_absorb_bmm(const mla_absorb_bmm_args& a, void* stream) {
  if (a.num_tokens == 0) return MLA_OK;
  EncodeTiledFn enc = encoder();
  if (!enc) return MLA_ERR_CUDA;
  const bool fp8 = a.w_dtype == MLA_W_FP8_E4M3;

  BmmParams p;
  p.out = reinterpret_cast<__nv_bfloat16*>(a.out);
  p.o_ts = a.out_stride_token;
  p.o_hs = a.out_stride_head;
  p.w_scale = a.w_scale;
  p.n_tok = a.num_tokens;
  p.H = a.num_heads;
  p.K = a.k;
  p.N = a.n;
  p.tok_tile = a.num_tokens >= 256 ? 256 : (a.num_tokens + 15) / 16 * 16;
  p.n_mtiles = a.n / 128;
  p.tmem_cols = pow2_at_least(p.tok_tile < 32 ? 32 : p.tok_tile);
  p.stage_bytes = kWTileBytes + p.tok_tile * 128 + (fp8 ? kWRawBytes : 0);
  p.status = a.status_d;
  const int nk = a.k / kKChunk;
  const int bar_bytes = (int)((sizeof(BmmBars) + 127) / 128 * 128);
  const int smem_cap = 227 * 1024 - kSmemAlign - bar_bytes;
  p.stages = nk < kMaxStages ? nk : kMaxStages;
  while (p.stages > 1 && p.stages * p.stage_bytes > smem_cap) --p.stages;
  if (p.stages * p.stage_bytes > smem_cap) return MLA_ERR_UNSUPPORTED;
  int smem = p.stages * p.stage_bytes + bar_bytes + kSmemAlign;
  // Never more CTAs on an SM than its 512 TMEM columns hold, so an allocation
  // never waits for another CTA: request enough shared memory to cap residency.
  const int max_ctas = 512 / p.tmem_cols;
  const int min_smem = 228 * 1024 / (max_ctas + 1) + 1024;
  if (smem < min_smem) smem = min_smem;

  CUtensorMap tx, tw;
  {
    const cuuint64_t gdim[3] = {(cuuint64_t)a.k, (cuuint64_t)a.num_heads, (cuuint64_t)a.num_tokens};
    const cuuint64_t gstride[2] = {(cuuint64_t)a.x_stride_head * 2, (cuuint64_t)a.x_stride_token * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kKChunk, 1u, (cuuint32_t)p.tok_tile};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.x), gdim, gstride, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_INVALID_ARG;
  }
  {
    const int esz = fp8 ? 1 : 2;
    const cuuint64_t gdim[3] = {(cuuint64_t)a.n, (cuuint64_t)a.k, (cuuint64_t)a.num_heads};
    const cuuint64_t gstride[2] = {(cuuint64_t)a.n * esz, (cuuint64_t)a.n * a.k * esz};
    const cuuint32_t box[3] = {fp8 ? 128u : 64u, (cuuint32_t)kKChunk, 1u};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tw, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.w),
            gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_INVALID_ARG;
  }
  const int n_ttiles = (a.num_tokens + p.tok_tile - 1) / p.tok_tile;
  const dim3 grid((unsigned)(p.n_mtiles * n_ttiles), (unsigned)a.num_heads, 1);
  // The shared-memory limit is raised once per kernel (to the largest size any
  // call needs), outside stream capture in the usual first-call-then-capture order.
  static int smem_set[2] = {0, 0};
  auto kern = fp8 ? mla_absorb_bmm_kernel<true> : mla_absorb_bmm_kernel<false>;
  if (smem > smem_set[fp8]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MLA_ERR_CUDA;
    smem_set[fp8] = smem;
  }
  kern<<<grid, kThreads, smem, (cudaStream_t)stream>>>(tx, tw, p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
