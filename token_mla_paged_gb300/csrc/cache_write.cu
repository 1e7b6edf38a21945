// KV-cache write: new tokens' latent (512) and RoPE (64) columns -> one
// 576-wide pool row each, bf16 or fp8 e4m3fn with the per-tensor scale
// ("[ROCm] Dspark MLA module", Details: the decode KV-cache write,
// concat_and_cache_mla).  Every input has an explicit dtype and is converted,
// never reinterpreted (the same page reports an fp32 k_pe read as bf16 here).
//
// HBM-bound scatter: a warp per two tokens, each lane handles groups of 8 columns
// (16-byte bf16 loads or two 16-byte fp32 loads; 16-byte bf16 or 8-byte fp8
// stores), so every row is read and written with whole-sector accesses.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace mla {
namespace {

constexpr int kGroups = kDqk / 8;        // 72 groups of 8 columns per row
constexpr int kGroupsC = 512 / 8;        // the first 64 come from kv_c

struct CacheWriteParams {
  const void* kv_c;
  const void* k_pe;
  int64_t kv_c_stride, k_pe_stride;      // elements
  int kv_c_fp32, k_pe_fp32;
  const int32_t* slot_mapping;
  int64_t num_tokens, num_slots;
  void* pool;
  int pool_fp8;
  float inv_scale;                       // fp32 reciprocal of kv_scale (fp8 pool)
};

// 8 consecutive input values starting at `col` of row n, as loaded: one 16-byte
// word of bf16 (a) or two of fp32 (a, b).
template <bool kF32>
struct Raw8 {
  uint4 a, b;
};
template <>
struct Raw8<false> {
  uint4 a;
};
template <bool kF32>
__device__ __forceinline__ Raw8<kF32> load8(const void* base, int64_t stride, int64_t n, int col) {
  Raw8<kF32> r;
  if constexpr (kF32) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const float*>(base) + n * stride + col);
    r.a = __ldg(src);
    r.b = __ldg(src + 1);
  } else {
    r.a = __ldg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + n * stride + col));
  }
  return r;
}
// ... widened to float32 (bf16 widens exactly).
template <bool kF32>
__device__ __forceinline__ void widen8(const Raw8<kF32>& r, float (&v)[8]) {
  if constexpr (kF32) {
    v[0] = __uint_as_float(r.a.x); v[1] = __uint_as_float(r.a.y); v[2] = __uint_as_float(r.a.z); v[3] = __uint_as_float(r.a.w);
    v[4] = __uint_as_float(r.b.x); v[5] = __uint_as_float(r.b.y); v[6] = __uint_as_float(r.b.z); v[7] = __uint_as_float(r.b.w);
  } else {
    const uint32_t w[4] = {r.a.x, r.a.y, r.a.z, r.a.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      v[2 * k] = __uint_as_float(w[k] << 16);
      v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
    }
  }
}

// Two float32 values -> two e4m3fn bytes (lo at the lower address): round to
// nearest even, saturating to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}

// One row group: 8 columns of the token's row to the pool.
template <bool kFp8>
__device__ __forceinline__ void store8(const CacheWriteParams& p, int32_t slot, int grp, const float (&v)[8]) {
  if constexpr (kFp8) {
    float y[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = __fmul_rn(v[k], p.inv_scale);
    uint2 o;
    o.x = e4m3x2(y[0], y[1]) | (e4m3x2(y[2], y[3]) << 16);
    o.y = e4m3x2(y[4], y[5]) | (e4m3x2(y[6], y[7]) << 16);
    *reinterpret_cast<uint2*>(static_cast<uint8_t*>(p.pool) + (int64_t)slot * kDqk + 8 * grp) = o;
  } else {
    uint4 o;
    o.x = pack_bf16x2(v[0], v[1]);
    o.y = pack_bf16x2(v[2], v[3]);
    o.z = pack_bf16x2(v[4], v[5]);
    o.w = pack_bf16x2(v[6], v[7]);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.pool) + (int64_t)slot * kDqk + 8 * grp) = o;
  }
}

// A warp takes two tokens per step; each lane loads its (up to) three groups of
// both before storing any, so six 16-byte words per lane (twelve for fp32
// inputs) are in flight.  Instantiated per input and pool dtype.
template <bool kF32C, bool kF32PE, bool kFp8>
__global__ void __launch_bounds__(256, (kF32C || kF32PE) ? 2 : 4) mla_cache_write_kernel(const CacheWriteParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  const int64_t w0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int64_t n0 = 2 * w0; n0 < p.num_tokens; n0 += 2 * warps) {
    int32_t slot[2];
    Raw8<kF32C> c[2][2];       // groups lane and lane + 32 (latent columns)
    Raw8<kF32PE> e[2];         // group lane + 64 (RoPE columns, lanes 0-7)
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      const int64_t n = n0 + t;
      slot[t] = n < p.num_tokens ? __ldg(p.slot_mapping + n) : -1;
      if (slot[t] >= p.num_slots) slot[t] = -1;       // outside the pool: skipped like padding
      if (slot[t] < 0) continue;
      c[t][0] = load8<kF32C>(p.kv_c, p.kv_c_stride, n, 8 * lane);
      c[t][1] = load8<kF32C>(p.kv_c, p.kv_c_stride, n, 8 * (lane + 32));
      if (lane < kGroups - kGroupsC) e[t] = load8<kF32PE>(p.k_pe, p.k_pe_stride, n, 8 * lane);
    }
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      if (slot[t] < 0) continue;
      float f[8];
      widen8<kF32C>(c[t][0], f);
      store8<kFp8>(p, slot[t], lane, f);
      widen8<kF32C>(c[t][1], f);
      store8<kFp8>(p, slot[t], lane + 32, f);
      if (lane < kGroups - kGroupsC) {
        widen8<kF32PE>(e[t], f);
        store8<kFp8>(p, slot[t], kGroupsC + lane, f);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// Fused decode RoPE + q concat + cache write ("[ROCm] Dspark MLA module":
// fused_qk_rope_concat_and_cache_mla, decode RoPE + cache after absorb).

struct RopeParams {
  const uint16_t* q_nope;
  int64_t qn_tok, qn_head;               // element strides
  const uint16_t* q_pe;
  int64_t qp_tok, qp_head;
  uint16_t* q_out;                       // [n, H, 576]
  int num_heads;
  const uint16_t* kv_c;
  int64_t kv_c_stride;
  const uint16_t* k_pe;
  int64_t k_pe_stride;
  const int32_t* positions;
  const float* cos_sin;                  // [max_pos, 64]
  int64_t max_pos;
  int style;                             // MLA_ROPE_NEOX | MLA_ROPE_INTERLEAVED
  const int32_t* slot_mapping;
  int64_t num_tokens, num_slots;
  void* pool;
  float inv_scale;
};

// y_a = a*c - b*s, y_b = b*c + a*s, every product and sum rounded on its own.
__device__ __forceinline__ void rot(float a, float b, float c, float sn, float& ya, float& yb) {
  ya = __fsub_rn(__fmul_rn(a, c), __fmul_rn(b, sn));
  yb = __fadd_rn(__fmul_rn(b, c), __fmul_rn(a, sn));
}

__device__ __forceinline__ void widen_bf16x8(const uint4& u, float (&v)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    v[2 * k] = __uint_as_float(w[k] << 16);
    v[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ uint4 pack_bf16x8(const float (&v)[8]) {
  return make_uint4(pack_bf16x2(v[0], v[1]), pack_bf16x2(v[2], v[3]), pack_bf16x2(v[4], v[5]),
                    pack_bf16x2(v[6], v[7]));
}

// Rotate the 64 RoPE values held as 16-byte units (8 values each) by the lanes
// that own them.  neox: lane l < 4 owns units l and l + 4 (values 8l.. and
// 32 + 8l.., the halves that pair up); interleaved: lane l < 8 owns unit l
// (four adjacent pairs).  Unit k of the rotated row is written to out(k).
template <typename Out>
__device__ __forceinline__ void rope_row(const uint16_t* src, int lane, int style, const float* cs, Out out) {
  if (style == MLA_ROPE_NEOX) {
    if (lane < 4) {
      float a[8], b[8], ya[8], yb[8];
      widen_bf16x8(__ldg(reinterpret_cast<const uint4*>(src) + lane), a);
      widen_bf16x8(__ldg(reinterpret_cast<const uint4*>(src) + lane + 4), b);
#pragma unroll
      for (int k = 0; k < 8; ++k) rot(a[k], b[k], __ldg(cs + 8 * lane + k), __ldg(cs + 32 + 8 * lane + k), ya[k], yb[k]);
      out(lane, ya);
      out(lane + 4, yb);
    }
  } else {
    if (lane < 8) {
      float x[8], y[8];
      widen_bf16x8(__ldg(reinterpret_cast<const uint4*>(src) + lane), x);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        rot(x[2 * k], x[2 * k + 1], __ldg(cs + 4 * lane + k), __ldg(cs + 32 + 4 * lane + k), y[2 * k], y[2 * k + 1]);
      out(lane, y);
    }
  }
}

template <bool kFp8>
__global__ void __launch_bounds__(256) mla_rope_q_cache_kernel(const RopeParams p) {
  const int lane = threadIdx.x & 31;
  const int64_t nq = p.num_tokens * p.num_heads;
  const int64_t items = nq + p.num_tokens;
  const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
  for (int64_t it = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); it < items; it += warps) {
    const int64_t n = it < nq ? it / p.num_heads : it - nq;
    int64_t pos = __ldg(p.positions + n);
    pos = pos < 0 ? 0 : (pos >= p.max_pos ? p.max_pos - 1 : pos);   // outside the table: clamp
    const float* cs = p.cos_sin + pos * 64;
    if (it < nq) {
      // q row: 512 absorbed latent columns copied, 64 RoPE columns rotated, one 576-wide row
      const int h = (int)(it - n * p.num_heads);
      const uint4* qn = reinterpret_cast<const uint4*>(p.q_nope + n * p.qn_tok + h * p.qn_head);
      uint4* qo = reinterpret_cast<uint4*>(p.q_out + (n * p.num_heads + h) * kDqk);
      const uint4 u0 = __ldg(qn + lane), u1 = __ldg(qn + lane + 32);
      qo[lane] = u0;
      qo[lane + 32] = u1;
      rope_row(p.q_pe + n * p.qp_tok + h * p.qp_head, lane, p.style, cs,
                  [&](int k, const float (&v)[8]) { qo[64 + k] = pack_bf16x8(v); });
    } else {
      // cache row: kv_c and the rotated k_pe, encoded like mla_cache_write
      const int32_t slot = __ldg(p.slot_mapping + n);
      if (slot < 0 || slot >= p.num_slots) continue;
      CacheWriteParams cw;
      cw.pool = p.pool;
      cw.inv_scale = p.inv_scale;
      const uint4* kc = reinterpret_cast<const uint4*>(p.kv_c + n * p.kv_c_stride);
      float f[8];
      widen_bf16x8(__ldg(kc + lane), f);
      store8<kFp8>(cw, slot, lane, f);
      widen_bf16x8(__ldg(kc + lane + 32), f);
      store8<kFp8>(cw, slot, lane + 32, f);
      rope_row(p.k_pe + n * p.k_pe_stride, lane, p.style, cs,
                     [&](int k, const float (&v)[8]) { store8<kFp8>(cw, slot, kGroupsC + k, v); });
    }
  }
}

}  // namespace

mla_status launch_cache_write(const mla_cache_write_args& a, void* stream) {
  CacheWriteParams p;
  p.kv_c = a.kv_c;
  p.k_pe = a.k_pe;
  p.kv_c_stride = a.kv_c_stride;
  p.k_pe_stride = a.k_pe_stride;
  p.kv_c_fp32 = a.kv_c_dtype == MLA_ACT_FP32;
  p.k_pe_fp32 = a.k_pe_dtype == MLA_ACT_FP32;
  p.slot_mapping = a.slot_mapping;
  p.num_tokens = a.num_tokens;
  p.num_slots = a.num_slots;
  p.pool = a.kv_pool;
  p.pool_fp8 = a.kv_dtype == MLA_KV_FP8_E4M3;
  p.inv_scale = p.pool_fp8 ? 1.0f / a.kv_scale : 1.0f;
  if (a.num_tokens == 0) return MLA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  // 16 tokens per 256-thread block (two per warp); up to 4 resident blocks per SM,
  // then grid-stride
  const int64_t blocks_needed = (a.num_tokens + 15) / 16;
  const int64_t cap = (int64_t)sms * 4;
  const int blocks = (int)(blocks_needed < cap ? blocks_needed : cap);
  const int sel = (p.kv_c_fp32 ? 4 : 0) | (p.k_pe_fp32 ? 2 : 0) | (p.pool_fp8 ? 1 : 0);
  static void (*const kernels[8])(const CacheWriteParams) = {
      mla_cache_write_kernel<false, false, false>, mla_cache_write_kernel<false, false, true>,
      mla_cache_write_kernel<false, true, false>,  mla_cache_write_kernel<false, true, true>,
      mla_cache_write_kernel<true, false, false>,  mla_cache_write_kernel<true, false, true>,
      mla_cache_write_kernel<true, true, false>,   mla_cache_write_kernel<true, true, true>};
  kernels[sel]<<<blocks, 256, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

mla_status launch_rope_q_cache(const mla_rope_q_cache_args& a, void* stream) {
  RopeParams p;
  p.q_nope = static_cast<const uint16_t*>(a.q_nope);
  p.qn_tok = a.q_nope_stride_token;
  p.qn_head = a.q_nope_stride_head;
  p.q_pe = static_cast<const uint16_t*>(a.q_pe);
  p.qp_tok = a.q_pe_stride_token;
  p.qp_head = a.q_pe_stride_head;
  p.q_out = static_cast<uint16_t*>(a.q_out);
  p.num_heads = a.num_heads;
  p.kv_c = static_cast<const uint16_t*>(a.kv_c);
  p.kv_c_stride = a.kv_c_stride;
  p.k_pe = static_cast<const uint16_t*>(a.k_pe);
  p.k_pe_stride = a.k_pe_stride;
  p.positions = a.positions;
  p.cos_sin = a.cos_sin;
  p.max_pos = a.max_pos;
  p.style = a.rope_style;
  p.slot_mapping = a.slot_mapping;
  p.num_tokens = a.num_tokens;
  p.num_slots = a.num_slots;
  p.pool = a.kv_pool;
  const bool fp8 = a.kv_dtype == MLA_KV_FP8_E4M3;
  p.inv_scale = fp8 ? 1.0f / a.kv_scale : 1.0f;
  if (a.num_tokens == 0) return MLA_OK;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MLA_ERR_CUDA;
  const int64_t items = a.num_tokens * ((int64_t)a.num_heads + 1);
  const int64_t blocks_needed = (items + 7) / 8;
  const int64_t cap = (int64_t)sms * 8;
  const int blocks = (int)(blocks_needed < cap ? blocks_needed : cap);
  if (fp8) mla_rope_q_cache_kernel<true><<<blocks, 256, 0, (cudaStream_t)stream>>>(p);
  else mla_rope_q_cache_kernel<false><<<blocks, 256, 0, (cudaStream_t)stream>>>(p);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}

}  // namespace mla
