// Device-side helpers shared by the decode kernels: error recording, storage
// decoders, plan/item geometry and the visibility rule.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "mla_internal.h"

namespace mla {

__device__ __forceinline__ void record_error(int32_t* hdr, int code, int info) {
  if (atomicCAS(&hdr[kWsErrCode], 0, code) == 0) atomicExch(&hdr[kWsErrInfo], info);
}

__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// fp8 e4m3fn -> float, exact, from the format definition: sign, 4-bit exponent
// with bias 7, 3-bit mantissa; exponent 0 is subnormal (m * 2^-9); 0x7F/0xFF NaN.
__device__ __forceinline__ float e4m3_bits_to_float(uint32_t b) {
  const uint32_t e = (b >> 3) & 0xFu, m = b & 7u;
  float v = e == 0 ? (float)m * 0.001953125f : __uint_as_float(((e + 120u) << 23) | (m << 20));
  if ((b & 0x7Fu) == 0x7Fu) v = __uint_as_float(0x7FC00000u);
  return __uint_as_float(__float_as_uint(v) | ((b & 0x80u) << 24));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// Does the plan header agree with the call's parameters?
__device__ __forceinline__ bool plan_header_ok(const int32_t* plan, const DecodeParams& p) {
  return plan[kHMagic] == kPlanMagic && plan[kHVersion] == kPlanVersion &&
         plan[kHBatch] == p.batch && plan[kHHeads] == p.num_heads &&
         plan[kHMaxQ] == p.max_q_len && plan[kHWorkers] == p.num_workers &&
         plan[kHMode] == p.mode && plan[kHItemsCap] == p.items_cap &&
         plan[kHNItems] >= 0 && plan[kHNItems] <= p.items_cap;
}

// One work item: rows [row0, row0+nrows) of request b (row r = t*H + h), KV
// entries [e0, e1) of split s of S.
struct Item {
  int b, s, S, g, slot, group;
  int row0, nrows, T, L;
  int64_t q_row_base;   // global row index (token*H + head) of request row 0
  int64_t kv_off;       // kv_indptr[b]
  int e0, e1;           // entry range after the causal trim
  int64_t base, Lg;     // global position of entry 0; global length
  int stride;
  bool ok;
};

// Entry range of split s of S over a request of real length L: tiles
// [floor(s*N/S), floor((s+1)*N/S)) with N = ceil(L/64), clamped to L.
__device__ __forceinline__ void split_range(int s, int S, int L, int& e0, int& e1) {
  const int64_t N = (L + kBlockN - 1) / kBlockN;
  const int64_t t0 = (int64_t)s * N / S, t1 = (int64_t)(s + 1) * N / S;
  e0 = (int)(t0 * kBlockN);
  e1 = (int)(t1 * kBlockN < (int64_t)L ? t1 * kBlockN : (int64_t)L);
}

__device__ __forceinline__ Item load_item(const DecodeParams& p, int idx) {
  Item it;
  const int32_t* plan = p.plan;
  const int B = p.batch;
  const int64_t off_S = kPlanHeaderInts, off_g = off_S + B, off_p = off_g + B + 1,
                off_i = off_p + B;
  const int32_t* rec = plan + off_i + 4LL * idx;
  it.b = rec[0];
  it.s = rec[1];
  it.g = rec[2];
  it.slot = rec[3];
  it.ok = it.b >= 0 && it.b < B;
  if (!it.ok) return it;
  const int b = it.b;
  it.S = plan[off_S + b];
  const int G = plan[off_g + b + 1] - plan[off_g + b];
  it.group = plan[off_g + b] + it.g;
  const int q0 = p.qo_indptr[b], q1 = p.qo_indptr[b + 1];
  it.T = q1 - q0;
  const int Gact = it.T > 0 ? (int)(((int64_t)it.T * p.num_heads + kRows - 1) / kRows) : 0;
  if (it.T < 0 || Gact != G || it.s < 0 || it.s >= it.S || it.g < 0 || it.g >= G) {
    record_error(p.ws_hdr, MLA_DEV_ROWS_MISMATCH, b);
    it.ok = false;
    return it;
  }
  int L = p.kv_indptr[b + 1] - p.kv_indptr[b];
  if (L < 0) {
    record_error(p.ws_hdr, MLA_DEV_BAD_INDPTR, b);
    L = 0;
  }
  it.L = L;
  it.kv_off = p.kv_indptr[b];
  it.q_row_base = (int64_t)q0 * p.num_heads;
  it.row0 = it.g * kRows;
  it.nrows = min(kRows, it.T * p.num_heads - it.row0);
  split_range(it.s, it.S, L, it.e0, it.e1);
  it.base = p.pos_base_per_req ? (int64_t)p.pos_base_per_req[b] : (int64_t)p.pos_base;
  it.Lg = p.g_kv_indptr ? (int64_t)(p.g_kv_indptr[b + 1] - p.g_kv_indptr[b]) : (int64_t)L;
  it.stride = p.pos_stride;
  if (p.causal) {
    // The group's last token sees the most; entries past its limit are masked for all rows.
    const int t_hi = (it.row0 + it.nrows - 1) / p.num_heads;
    const int64_t lim_abs = it.Lg - it.T + t_hi;
    int64_t count;
    if (p.kv_pos) {
      // positions ascend within a request: count those <= the limit
      int64_t lo = 0, hi = L;
      while (lo < hi) {
        const int64_t mid = (lo + hi) >> 1;
        if ((int64_t)p.kv_pos[it.kv_off + mid] <= lim_abs) lo = mid + 1;
        else hi = mid;
      }
      count = lo;
    } else {
      const int64_t lim = lim_abs - it.base;
      count = lim < 0 ? 0 : lim / it.stride + 1;
    }
    if ((int64_t)it.e1 > count) it.e1 = (int)(count > (int64_t)it.e0 ? count : (int64_t)it.e0);
  }
  return it;
}

// Global position of local entry i.
__device__ __forceinline__ int64_t entry_pos(const Item& it, const DecodeParams& p, int64_t i) {
  return p.kv_pos ? (int64_t)p.kv_pos[it.kv_off + i] : it.base + i * it.stride;
}

// Visibility of local entry i for token t: causal limit Lg - T + t and, with a
// window W > 0, positions above limit - W.
__device__ __forceinline__ bool visible(const Item& it, const DecodeParams& p, int64_t i, int t) {
  if (!p.causal) return true;
  const int64_t lim = it.Lg - it.T + t, g = entry_pos(it, p, i);
  return g <= lim && (p.window <= 0 || g > lim - p.window);
}

}  // namespace mla
