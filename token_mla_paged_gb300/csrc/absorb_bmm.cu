// Absorb BMMs either side of the latent decode ("[ROCm] Dspark MLA module",
// Details: the decode's absorb BMM, FP8/FP4 BMM when enabled, else torch.bmm):
//   before: q_lat[t, h, :] = q_nope[t, h, :] @ W_UK[h]     (k = 128, n = 512)
//   after:  out[t, h, :]   = o_lat[t, h, :]  @ W_UV[h]     (k = 512, n = 128)
// One kernel computes y[t, h, j] = bf16(s * sum_k x[t, h, k] * w[h, k, j]).
//
// The work is HBM-bound (each weight byte and each activation byte is used a few
// hundred times at most), so the kernel is built to keep every SM streaming:
//   * a unit is (head, 128 tokens, 128 output columns); one persistent CTA per
//     SM walks its units in a fixed stride;
//   * per 64-wide k chunk TMA brings the token tile [128 t][64 k] (bf16, 128-byte
//     swizzled: the K-major A operand, rows past the last token zero-filled) and
//     the weight tile [64 k][128 j] (bf16 as 64-column swizzled boxes: the
//     MN-major B operand; fp8 as one raw box that eight conversion warps expand
//     exactly to bf16 in that same layout), through a ring of stages that runs
//     across unit boundaries;
//   * four tcgen05.mma (M=128, N=128, K=16) per chunk accumulate D[t, j] in one
//     of two TMEM accumulators, so the epilogue of a unit overlaps the loads and
//     MMAs of the next;
//   * each epilogue warp owns 32 token rows x 64 columns: TMEM -> registers, times s,
//     rounded to bf16, staged in 2 KB of XOR-swizzled shared memory per warp and
//     written as whole 64-byte row segments.
// Warp roles: 0 TMA producer, 1 TMEM allocation + MMA issue, 2-9 epilogue (two
// per TMEM lane quadrant, 64 columns each), 10-17 fp8 conversion (fp8 only).  Every barrier wait is bounded; a wait
// that runs out records MLA_DEV_WAIT_TIMEOUT (and the wait site) in the optional
// status word and raises an abort flag; the CTA then lets its copies and MMAs in
// flight complete (bounded waits again), frees TMEM and returns.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "mla_internal.h"
#include "tc_primitives.cuh"

namespace mla {
namespace {

using namespace tc;

constexpr int kKChunk = 64;                   // k per pipeline stage
constexpr int kTokTile = 128;                 // M of the MMA
constexpr int kNTile = 128;                   // N of the MMA: output columns per unit
constexpr int kXBytes = kTokTile * 128;       // token tile per chunk (16 KB)
constexpr int kWBlockBytes = 64 * 128;        // bf16 weight block [64 k][64 j]
constexpr int kMaxStages = 6;
constexpr int kSmemAlign = 1024;
constexpr int kEpiWarps = 8;                  // two per TMEM lane quadrant, 64 columns each
constexpr int kEpiBytes = kEpiWarps * 2048;   // per-warp staging of the epilogue

constexpr int kConvWarps = 8;                 // fp8 weight conversion
__host__ __device__ constexpr int threads_for(bool fp8) { return 32 * (2 + kEpiWarps + (fp8 ? kConvWarps : 0)); }

struct BmmParams {
  __nv_bfloat16* out;
  long long o_ts, o_hs;  // elements
  float w_scale;
  int n_tok, H, K, N;
  int stages;            // 2..kMaxStages
  int n_ttiles, n_jtiles, units;
  int stage_bytes;       // token tile + bf16 weight tile (+ raw fp8 tile)
  int32_t* status;       // optional
};

struct BmmBars {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t conv[kMaxStages];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
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

// Two e4m3fn codes (low byte first) -> two bf16 values, exactly.  e4m3 -> f16
// is exact (one conversion instruction for the pair); every such f16 has at
// most 3 significant mantissa bits and is normal (e4m3's subnormals are f16
// normals), so the bf16 keeps the sign, drops the 3 low mantissa bits and
// re-biases the exponent from 15 to 127 (+112); zeros stay zero.  The NaN codes
// 0x7F / 0xFF are outside the contract (they come out finite).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(two));
  const uint32_t mag = h & 0x7FFF7FFFu;
  const uint32_t bias = ((mag & 0xFFFFu) ? 0x3800u : 0u) | ((mag >> 16) ? 0x38000000u : 0u);
  return (((mag >> 3) & 0x0FFF0FFFu) + bias) | (h & 0x80008000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ void record_timeout(const BmmParams& p, volatile int* abort, int site) {
  if (p.status && atomicCAS(p.status, 0, (int32_t)MLA_DEV_WAIT_TIMEOUT) == 0) p.status[1] = site;
  *abort = 1;
}

struct Unit {
  int h, t0, j0;
};
__device__ __forceinline__ Unit unit_of(const BmmParams& p, int u) {
  Unit r;
  r.h = u / (p.n_ttiles * p.n_jtiles);
  const int rem = u - r.h * (p.n_ttiles * p.n_jtiles);
  r.t0 = (rem / p.n_jtiles) * kTokTile;
  r.j0 = (rem % p.n_jtiles) * kNTile;
  return r;
}

// Bounded wait in which the thread sleeps in the barrier until the phase
// completes (or 0.5 ms pass) instead of spinning, so waiting warps leave the
// shared-memory pipe to the warps that work.  Gives up after about a second, or
// when *abort is set.
__device__ __forceinline__ bool try_wait_suspend(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(500000u)
      : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_phase(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (try_wait_suspend(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    if (try_wait_suspend(bar, parity)) return true;
    if (*abort) return false;
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
}

#define BMM_WAIT(bar, parity, site, label)                   \
  if (!wait_phase((bar), (parity), abort)) {                 \
    if (!*abort) record_timeout(p, abort, (site));           \
    goto label;                                              \
  }

template <bool kFp8>
__global__ void __launch_bounds__(threads_for(kFp8), 1)
    mla_absorb_bmm_kernel(const __grid_constant__ CUtensorMap tmap_x, const __grid_constant__ CUtensorMap tmap_w,
                          const BmmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + kSmemAlign - 1) & ~(uintptr_t)(kSmemAlign - 1));
  uint8_t* epi = smem + p.stages * p.stage_bytes;
  BmmBars* bars = reinterpret_cast<BmmBars*>(epi + kEpiBytes);
  volatile int* abort = &bars->abort;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nk = p.K / kKChunk;
  const int wbytes = kNTile * 128;             // bf16 weight tile per chunk
  const int nblk = kNTile / 64;

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&bars->full[s], 1);
      mbar_init(&bars->empty[s], 1);
      mbar_init(&bars->conv[s], 32 * kConvWarps);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars->acc_full[b], 1);
      mbar_init(&bars->acc_empty[b], 32 * kEpiWarps);
    }
    mbar_init(&bars->drain, 1);
    bars->abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_x);
    prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_slot, (uint32_t)(2 * kNTile));
    tmem_relinquish();
  }
  fence_before_sync();
  __syncthreads();
  fence_after_sync();
  const uint32_t tmem = bars->tmem_slot;
  const uint32_t sbase = smem_u32(smem);
  // The set-up above overlaps the end of the previous kernel on the stream; the
  // activations it may have written are read only after this wait.
  grid_dependency_wait();
  allow_dependent_launch();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t g = 0, issued_from = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        const Unit un = unit_of(p, u);
        for (int c = 0; c < nk; ++c, ++g) {
          const int s = (int)(g % p.stages);
          BMM_WAIT(&bars->empty[s], ((g / p.stages) & 1) ^ 1, 1, done_producer);
          const uint32_t st = sbase + (uint32_t)(s * p.stage_bytes);
          mbar_arrive_expect_tx(&bars->full[s], (uint32_t)(kXBytes + (kFp8 ? kNTile * kKChunk : wbytes)));
          tma_load_3d(st, &tmap_x, c * kKChunk, un.h, un.t0, &bars->full[s]);
          if (kFp8) {
            tma_load_3d(st + kXBytes + wbytes, &tmap_w, un.j0, c * kKChunk, un.h, &bars->full[s]);
          } else {
            for (int b = 0; b < nblk; ++b)
              tma_load_3d(st + kXBytes + b * kWBlockBytes, &tmap_w, un.j0 + 64 * b, c * kKChunk, un.h,
                          &bars->full[s]);
          }
        }
      }
    done_producer:
      if (*abort) {
        // Let the copies already issued land before the shared memory goes away.
        issued_from = g > (uint32_t)p.stages ? g - p.stages : 0;
        for (uint32_t c = issued_from; c < g; ++c) {
          const long long t0c = clock64();
          while (!mbar_try_wait(&bars->full[c % p.stages], (c / p.stages) & 1) &&
                 clock64() - t0c < kWaitLimitCycles) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(kTokTile, kNTile, false, true);
      uint32_t g = 0, i = 0;
      bool any = false;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
        const uint32_t buf = i & 1;
        BMM_WAIT(&bars->acc_empty[buf], ((i >> 1) & 1) ^ 1, 2, done_mma);
        fence_after_sync();
        for (int c = 0; c < nk; ++c, ++g) {
          const int s = (int)(g % p.stages);
          BMM_WAIT(kFp8 ? &bars->conv[s] : &bars->full[s], (g / p.stages) & 1, 3, done_mma);
          fence_after_sync();
          const uint32_t st = sbase + (uint32_t)(s * p.stage_bytes);
          const uint64_t adesc = smem_desc_sw128(st, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(st + kXBytes, kWBlockBytes, 1024);
#pragma unroll
          for (int k = 0; k < kKChunk / 16; ++k)
            mma_ss(tmem + buf * (uint32_t)kNTile, adesc + (uint64_t)((k * 32) >> 4),
                   bdesc + (uint64_t)((k * 2048) >> 4), idesc, (c > 0 || k > 0) ? 1u : 0u);
          mma_commit(&bars->empty[s]);
          any = true;
        }
        mma_commit(&bars->acc_full[buf]);
      }
    done_mma:
      if (*abort && any) {
        mma_commit(&bars->drain);
        const long long t0c = clock64();
        while (!mbar_try_wait(&bars->drain, 0) && clock64() - t0c < kWaitLimitCycles) {
        }
      }
    }
    __syncwarp();
  } else if (warp < 2 + kEpiWarps) {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;                   // TMEM lanes = token rows 32*quad .. +31
    const int half = (warp - 2) >> 2;            // columns 64*half .. +63
    uint8_t* stg = epi + (warp - 2) * 2048;
    uint32_t i = 0;
    for (int u = blockIdx.x; u < p.units; u += gridDim.x, ++i) {
      const Unit un = unit_of(p, u);
      const uint32_t buf = i & 1;
      BMM_WAIT(&bars->acc_full[buf], (i >> 1) & 1, 4, done_epilogue);
      fence_after_sync();
      uint32_t acc[2][32];
      {
        const uint32_t ta = tmem + buf * (uint32_t)kNTile + ((uint32_t)(32 * quad) << 16) + 64 * half;
        tmem_ld32(ta, acc[0]);
        tmem_ld32(ta + 32, acc[1]);
        tmem_wait_ld();
      }
      fence_before_sync();
      mbar_arrive(&bars->acc_empty[buf]);
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        const int c0 = 64 * half + 32 * g2;
        const uint32_t* r = acc[g2];
        // row `lane` of the staging block: 4 units of 8 columns, XOR-swizzled by row
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16x2(__uint_as_float(r[8 * q + 0]) * p.w_scale, __uint_as_float(r[8 * q + 1]) * p.w_scale);
          v.y = pack_bf16x2(__uint_as_float(r[8 * q + 2]) * p.w_scale, __uint_as_float(r[8 * q + 3]) * p.w_scale);
          v.z = pack_bf16x2(__uint_as_float(r[8 * q + 4]) * p.w_scale, __uint_as_float(r[8 * q + 5]) * p.w_scale);
          v.w = pack_bf16x2(__uint_as_float(r[8 * q + 6]) * p.w_scale, __uint_as_float(r[8 * q + 7]) * p.w_scale);
          *reinterpret_cast<uint4*>(stg + lane * 64 + ((q ^ ((lane >> 1) & 3)) << 4)) = v;
        }
        __syncwarp();
#pragma unroll
        for (int pass = 0; pass < 4; ++pass) {
          const int row = pass * 8 + (lane >> 2), q = lane & 3;
          const int t = un.t0 + 32 * quad + row;
          const uint4 v = *reinterpret_cast<const uint4*>(stg + row * 64 + ((q ^ ((row >> 1) & 3)) << 4));
          if (t < p.n_tok)
            *reinterpret_cast<uint4*>(p.out + (long long)t * p.o_ts + (long long)un.h * p.o_hs + un.j0 + c0 +
                                      8 * q) = v;
        }
        __syncwarp();
      }
    }
  done_epilogue:;
  } else {
    // ------------------------------------------------------------ fp8 conversion
    if (kFp8) {
      const int tid = threadIdx.x - 32 * (2 + kEpiWarps);   // 0 .. 32 * kConvWarps - 1
      constexpr int upr = kNTile / 8;            // 8-byte raw groups per k row
      constexpr int iters = kKChunk * upr / (32 * kConvWarps);
      uint32_t g = 0;
      for (int u = blockIdx.x; u < p.units; u += gridDim.x) {
        for (int c = 0; c < nk; ++c, ++g) {
          const int s = (int)(g % p.stages);
          BMM_WAIT(&bars->full[s], (g / p.stages) & 1, 5, done_convert);
          uint8_t* st = smem + s * p.stage_bytes + kXBytes;
          const uint8_t* raw = st + wbytes;
          // thread -> 8 consecutive columns of one k row: eight neighbouring threads
          // fill one 128-byte line of the swizzled tile, so the stores do not
          // conflict; all raw words are loaded first so the conversions overlap
          uint2 x[iters];
#pragma unroll
          for (int it = 0; it < iters; ++it) {
            const int v = tid + 32 * kConvWarps * it, kr = v / upr, col = (v - kr * upr) * 8;
            x[it] = *reinterpret_cast<const uint2*>(raw + kr * kNTile + col);
          }
#pragma unroll
          for (int it = 0; it < iters; ++it) {
            const int v = tid + 32 * kConvWarps * it, kr = v / upr, col = (v - kr * upr) * 8;
            const uint4 o = make_uint4(e4m3x2_to_bf16x2((uint16_t)(x[it].x & 0xFFFFu)),
                                       e4m3x2_to_bf16x2((uint16_t)(x[it].x >> 16)),
                                       e4m3x2_to_bf16x2((uint16_t)(x[it].y & 0xFFFFu)),
                                       e4m3x2_to_bf16x2((uint16_t)(x[it].y >> 16)));
            const int blk = col >> 6, uu = (col & 63) >> 3;   // 64-column block, unit in its line
            *reinterpret_cast<uint4*>(st + blk * kWBlockBytes + kr * 128 + ((uu ^ (kr & 7)) << 4)) = o;
          }
          fence_proxy_async_smem();
          mbar_arrive(&bars->conv[s]);
        }
      }
    done_convert:;
    }
  }

  fence_before_sync();
  __syncthreads();
  if (warp == 1) tmem_dealloc(tmem, (uint32_t)(2 * kNTile));
}

#undef BMM_WAIT

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

}  // namespace

mla_status launch_absorb_bmm(const mla_absorb_bmm_args& a, void* stream) {
  if (a.num_tokens == 0) return MLA_OK;
  EncodeTiledFn enc = encoder();
  const int dev = current_device_slot();
  const int sms = device_sm_count(dev);
  if (!enc || sms <= 0) return MLA_ERR_CUDA;
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
  p.n_ttiles = (a.num_tokens + kTokTile - 1) / kTokTile;
  p.n_jtiles = a.n / kNTile;
  const long long units = (long long)a.num_heads * p.n_ttiles * p.n_jtiles;
  if (units > 0x7FFFFFFFLL) return MLA_ERR_UNSUPPORTED;
  p.units = (int)units;
  p.stage_bytes = kXBytes + kNTile * 128 + (fp8 ? kNTile * kKChunk : 0);
  p.status = a.status_d;
  const int bar_bytes = (int)((sizeof(BmmBars) + 127) / 128 * 128);
  const int smem_cap = 227 * 1024 - kSmemAlign - kEpiBytes - bar_bytes;
  p.stages = kMaxStages;
  while (p.stages > 2 && p.stages * p.stage_bytes > smem_cap) --p.stages;
  if (p.stages * p.stage_bytes > smem_cap) return MLA_ERR_UNSUPPORTED;
  int smem = p.stages * p.stage_bytes + kEpiBytes + bar_bytes + kSmemAlign;
  // One CTA per SM (its ring fills the shared memory); the request never drops
  // below half the SM's shared memory, so two CTAs' accumulators (2 x 256 TMEM
  // columns) are the most an SM could ever be asked for.
  const int one_cta = 228 * 1024 / 2 + 1024;
  if (smem < one_cta) smem = one_cta;

  CUtensorMap tx, tw;
  {
    const cuuint64_t gdim[3] = {(cuuint64_t)a.k, (cuuint64_t)a.num_heads, (cuuint64_t)a.num_tokens};
    const cuuint64_t gstride[2] = {(cuuint64_t)a.x_stride_head * 2, (cuuint64_t)a.x_stride_token * 2};
    const cuuint32_t box[3] = {(cuuint32_t)kKChunk, 1u, (cuuint32_t)kTokTile};
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
    const cuuint32_t box[3] = {fp8 ? (cuuint32_t)kNTile : 64u, (cuuint32_t)kKChunk, 1u};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (enc(&tw, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(a.w),
            gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            fp8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return MLA_ERR_INVALID_ARG;
  }
  const int grid = p.units < sms ? p.units : sms;
  // The shared-memory limit is raised once per kernel (to the largest size any
  // call needs), outside stream capture in the usual first-call-then-capture order.
  static int smem_set[kMaxDevices][2] = {};
  auto kern = fp8 ? mla_absorb_bmm_kernel<true> : mla_absorb_bmm_kernel<false>;
  if (smem > smem_set[dev][fp8]) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
      return MLA_ERR_CUDA;
    smem_set[dev][fp8] = smem;
  }
  return launch_overlapped(kern, dim3(grid), dim3(threads_for(fp8)), smem, (cudaStream_t)stream, tx, tw, p) ==
                 cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace mla
