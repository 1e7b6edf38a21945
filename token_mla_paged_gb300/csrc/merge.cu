// N-way merge of partial attention states (O_s, LSE_s) over disjoint KV
// subsets, e.g. the per-shard results of round-robin context parallelism
// ("Speculative decode + DCP on gfx1250", Problem: a verify pass over a
// round-robin DCP shard with an LSE output).
//
//   M = max_s LSE_s;  LSE = M + ln sum_s exp(LSE_s - M);  O = sum_s exp(LSE_s - LSE) O_s
//
// One warp per row; lanes stride over the row's dv columns (coalesced).  For up
// to 32 states the per-state weights are computed once per row (one per lane)
// and broadcast with shuffles; more states recompute them per column block.
// The work is HBM-bound: n*dv reads and dv writes per row.
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace mla {
namespace {

__global__ void __launch_bounds__(256)
mla_merge_states_kernel(const void* __restrict__ o_parts, int parts_fp32,
                        const float* __restrict__ lse_parts, int n, int64_t rows, int dv,
                        void* __restrict__ o, int o_fp32, float* __restrict__ lse) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows;
       r += warps_total) {
    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, lse_parts[(int64_t)s * rows + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float tot = 0.f;
    if (M != -INFINITY) {
      for (int s = lane; s < n; s += 32) {
        const float ls = lse_parts[(int64_t)s * rows + r];
        if (ls != -INFINITY) tot += exp2f((ls - M) * 1.4426950408889634f);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    }
    const float inv_tot = M != -INFINITY ? 1.f / tot : 0.f;
    // Weight of state s: exp(LSE_s - M) / tot.  With n <= 32 lane s keeps state
    // s's weight in a register for the whole row; beyond that the weights of each
    // 32-state chunk are recomputed per column block.  Either way the states are
    // summed in order 0..n-1 for every column.
    const bool hoisted = n <= 32;
    float w_own = 0.f;
    if (hoisted && lane < n && M != -INFINITY) {
      const float ls = lse_parts[(int64_t)lane * rows + r];
      w_own = ls == -INFINITY ? 0.f : exp2f((ls - M) * 1.4426950408889634f) * inv_tot;
    }
    for (int d0 = 0; d0 < dv; d0 += 32) {
      const int d = d0 + lane;
      float acc = 0.f;
      if (M != -INFINITY) {
        for (int c = 0; c < n; c += 32) {
          float w = w_own;
          if (!hoisted) {
            w = 0.f;
            if (c + lane < n) {
              const float ls = lse_parts[(int64_t)(c + lane) * rows + r];
              w = ls == -INFINITY ? 0.f : exp2f((ls - M) * 1.4426950408889634f) * inv_tot;
            }
          }
          const int cnt = min(32, n - c);
          for (int k = 0; k < cnt; ++k) {
            const float wk = __shfl_sync(0xffffffffu, w, k);
            if (d < dv && wk != 0.f) {
              const int64_t off = ((int64_t)(c + k) * rows + r) * dv + d;
              const float v = parts_fp32 ? static_cast<const float*>(o_parts)[off]
                                         : bf16_bits_to_float(static_cast<const uint16_t*>(o_parts)[off]);
              acc += wk * v;
            }
          }
        }
      }
      if (d < dv) {
        if (o_fp32) static_cast<float*>(o)[r * dv + d] = acc;
        else static_cast<__nv_bfloat16*>(o)[r * dv + d] = __float2bfloat16_rn(acc);
      }
    }
    if (lane == 0) lse[r] = M == -INFINITY ? -INFINITY : M + logf(tot);
  }
}

// Fast path for the common shape: dv a multiple of 256 with 16-byte aligned
// rows (dv = 512 in every MLA call).  One warp per row as above, but lane l owns
// 8 consecutive columns of every 256-column block and reads them as one 16-byte
// (bf16) or two 16-byte (fp32) vectors per state, all states' loads issued
// before they are combined, so each lane has n loads in flight.  The states are
// summed in order 0..n-1, as in the general kernel.
template <bool kPartsF32, bool kOutF32, int kMaxN>
__global__ void __launch_bounds__(256)
mla_merge_states_vec_kernel(const void* __restrict__ o_parts, const float* __restrict__ lse_parts, int n,
                            int64_t rows, int dv, void* __restrict__ o, float* __restrict__ lse) {
  grid_dependency_wait();
  allow_dependent_launch();
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x / 32);
  for (int64_t r = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); r < rows; r += warps_total) {
    float M = -INFINITY;
    for (int s = lane; s < n; s += 32) M = fmaxf(M, lse_parts[(int64_t)s * rows + r]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
    float tot = 0.f;
    if (M != -INFINITY) {
      for (int s = lane; s < n; s += 32) {
        const float ls = lse_parts[(int64_t)s * rows + r];
        if (ls != -INFINITY) tot += exp2f((ls - M) * 1.4426950408889634f);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    }
    const float inv_tot = M != -INFINITY ? 1.f / tot : 0.f;
    // lane s (< n) holds state s's weight
    float w_own = 0.f;
    if (lane < n && M != -INFINITY) {
      const float ls = lse_parts[(int64_t)lane * rows + r];
      w_own = ls == -INFINITY ? 0.f : exp2f((ls - M) * 1.4426950408889634f) * inv_tot;
    }
    for (int d0 = 8 * lane; d0 < dv; d0 += 256) {
      float acc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) acc[k] = 0.f;
      float v[kMaxN][8];
#pragma unroll
      for (int s = 0; s < kMaxN; ++s) {
        if (s < n) {
          const int64_t off = ((int64_t)s * rows + r) * dv + d0;
          if (kPartsF32) {
            const float4 a = *reinterpret_cast<const float4*>(static_cast<const float*>(o_parts) + off);
            const float4 b = *reinterpret_cast<const float4*>(static_cast<const float*>(o_parts) + off + 4);
            v[s][0] = a.x; v[s][1] = a.y; v[s][2] = a.z; v[s][3] = a.w;
            v[s][4] = b.x; v[s][5] = b.y; v[s][6] = b.z; v[s][7] = b.w;
          } else {
            const uint4 a = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(o_parts) + off);
            const uint32_t w4[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              v[s][2 * k] = bf16_bits_to_float(w4[k] & 0xFFFFu);
              v[s][2 * k + 1] = bf16_bits_to_float(w4[k] >> 16);
            }
          }
        }
      }
#pragma unroll
      for (int s = 0; s < kMaxN; ++s) {
        if (s < n) {
          const float ws = __shfl_sync(0xffffffffu, w_own, s);
          if (ws != 0.f) {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] += ws * v[s][k];
          }
        }
      }
      if (kOutF32) {
        float* dst = static_cast<float*>(o) + r * dv + d0;
        *reinterpret_cast<float4*>(dst) = make_float4(acc[0], acc[1], acc[2], acc[3]);
        *reinterpret_cast<float4*>(dst + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
      } else {
        *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(o) + r * dv + d0) =
            make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                       pack_bf16x2(acc[6], acc[7]));
      }
    }
    if (lane == 0) lse[r] = M == -INFINITY ? -INFINITY : M + logf(tot);
  }
}

}  // namespace

mla_status launch_merge_states(const void* o_parts, int o_parts_fp32, const float* lse_parts,
                               int n, int64_t rows, int dv, void* o, int o_fp32, float* lse,
                               void* stream) {
  const int num_sms = device_sm_count(current_device_slot());
  if (num_sms == 0) return MLA_ERR_CUDA;
  const int64_t want = (rows + 7) / 8;
  const int grid = (int)(want < (int64_t)num_sms * 16 ? want : (int64_t)num_sms * 16);
  const bool vec = n <= 16 && dv % 256 == 0 && ((uintptr_t)o_parts % 16) == 0 && ((uintptr_t)o % 16) == 0;
  cudaStream_t st = (cudaStream_t)stream;
  if (vec) {
    // (states in registers: up to 8, else up to 16)
    auto pick = [&](auto k8, auto k16) { return n <= 8 ? k8 : k16; };
    void (*kern)(const void*, const float*, int, int64_t, int, void*, float*);
    if (o_parts_fp32 && o_fp32)
      kern = pick(mla_merge_states_vec_kernel<true, true, 8>, mla_merge_states_vec_kernel<true, true, 16>);
    else if (o_parts_fp32)
      kern = pick(mla_merge_states_vec_kernel<true, false, 8>, mla_merge_states_vec_kernel<true, false, 16>);
    else if (o_fp32)
      kern = pick(mla_merge_states_vec_kernel<false, true, 8>, mla_merge_states_vec_kernel<false, true, 16>);
    else
      kern = pick(mla_merge_states_vec_kernel<false, false, 8>, mla_merge_states_vec_kernel<false, false, 16>);
    return launch_overlapped(kern, dim3(grid), dim3(256), 0, st, o_parts, lse_parts, n, rows, dv, o, lse) ==
                   cudaSuccess
               ? MLA_OK
               : MLA_ERR_CUDA;
  }
  return launch_overlapped(mla_merge_states_kernel, dim3(grid), dim3(256), 0, st, o_parts, o_parts_fp32, lse_parts,
                           n, rows, dv, o, o_fp32, lse) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace mla
