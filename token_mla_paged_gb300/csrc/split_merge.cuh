// Fused split-merge epilogue: the last split of a (request, row group) to
// finish combines every split's partial (O, LSE) through the log-sum-exp and
// writes the final output.  Long rows are split over the KV and merged inside
// the same call ("[DSV4] Tuned ASM FP8 decode with split plans; HCA on aiter's
// persistent V4-NM kernel", Summary part 2: in-kernel split and merge).
//
// Determinism: partials are combined in split order, so the result does not
// depend on which split arrived last.
#pragma once

#include "device_common.cuh"

namespace mla {

// Store one row's final output: 4 consecutive dims starting at d (fp32 or bf16).
__device__ __forceinline__ void store_o4(const DecodeParams& p, int64_t row, int d, float4 v) {
  if (p.out_fp32) {
    *reinterpret_cast<float4*>(static_cast<float*>(p.o) + row * kDv + d) = v;
  } else {
    uint2 u;
    u.x = pack_bf16x2(v.x, v.y);
    u.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(p.o) + row * kDv + d) = u;
  }
}

// Called by every thread of the block after this split's partials are written.
// Returns true if this block performed the merge.
__device__ inline bool arrive_and_merge(const DecodeParams& p, const Item& it, int* s_flag) {
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const int prev = atomicAdd(&p.counters[it.group], 1);
    *s_flag = (prev == it.S - 1);
  }
  __syncthreads();
  if (!*s_flag) return false;
  __threadfence();
  const int G = p.plan[kPlanHeaderInts + p.batch + it.b + 1] - p.plan[kPlanHeaderInts + p.batch + it.b];
  const int pbase = p.plan[kPlanHeaderInts + 2 * p.batch + 1 + it.b];
  const int nvec = it.nrows * (kDv / 4);
  for (int v = threadIdx.x; v < nvec; v += blockDim.x) {
    const int r = v / (kDv / 4), d = (v % (kDv / 4)) * 4;
    float M = -INFINITY;
    for (int s = 0; s < it.S; ++s) {
      const int slot = pbase + s * G + it.g;
      M = fmaxf(M, __ldcg(p.part_lse + (int64_t)slot * kRows + r));
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float tot = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < it.S; ++s) {
        const int slot = pbase + s * G + it.g;
        const float ls = __ldcg(p.part_lse + (int64_t)slot * kRows + r);
        if (ls == -INFINITY) continue;
        const float w = exp2f((ls - M) * 1.4426950408889634f);
        const float4 o = __ldcg(reinterpret_cast<const float4*>(
            p.part_o + ((int64_t)slot * kRows + r) * kDv + d));
        tot += w;
        acc.x += w * o.x;
        acc.y += w * o.y;
        acc.z += w * o.z;
        acc.w += w * o.w;
      }
      const float inv = 1.f / tot;
      acc.x *= inv;
      acc.y *= inv;
      acc.z *= inv;
      acc.w *= inv;
    }
    const int64_t row = it.q_row_base + it.row0 + r;
    store_o4(p, row, d, acc);
    if (d == 0) p.lse[row] = M == -INFINITY ? -INFINITY : M + logf(tot);
  }
  if (threadIdx.x == 0) p.counters[it.group] = 0;
  return true;
}

}  // namespace mla
