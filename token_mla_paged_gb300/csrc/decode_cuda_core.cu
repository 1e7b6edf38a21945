// CUDA-core MLA decode kernel: the same operation, plan and workspace as the
// tensor-core kernel, computed with plain fp32 FMAs.  It exists to cross-check
// the tensor-core path and as the simplest correct implementation on sm_103a.
//
// Persistent blocks pull work items (request b, split s, row group g) from an
// atomic queue over the plan's cost-sorted item list.  An item's rows (up to
// 256) are processed as 32-row passes over the item's KV range; each pass keeps
// Q[32, 576] and one KV tile [32, 576] in shared memory as fp32, the running
// max/sum per row in registers and O[32, 512] spread over 256 threads.
#include <cuda_runtime.h>

#include "device_common.cuh"
#include "split_merge.cuh"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kSubRows = 32;
constexpr int kTile = 32;
constexpr int kStride = kDqk + 4;   // padded fp32 row: conflict-free float4 column reads

__device__ __forceinline__ void load_row_f32(const DecodeParams& p, int64_t slot, float* dst,
                                             int lane) {
  if (p.kv_fp8) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(p.kv) + slot * kDqk);
    for (int c = lane; c < kDqk / 16; c += 32) {
      const uint4 u = __ldg(src + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        float4 f;
        f.x = e4m3_bits_to_float(w[k] & 0xFF);
        f.y = e4m3_bits_to_float((w[k] >> 8) & 0xFF);
        f.z = e4m3_bits_to_float((w[k] >> 16) & 0xFF);
        f.w = e4m3_bits_to_float(w[k] >> 24);
        *reinterpret_cast<float4*>(dst + c * 16 + 4 * k) = f;
      }
    }
  } else {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.kv) + slot * kDqk);
    for (int c = lane; c < kDqk / 8; c += 32) {
      const uint4 u = __ldg(src + c);
      const uint32_t w[4] = {u.x, u.y, u.z, u.w};
      float4 a, b;
      a.x = bf16_bits_to_float(w[0] & 0xFFFF);
      a.y = bf16_bits_to_float(w[0] >> 16);
      a.z = bf16_bits_to_float(w[1] & 0xFFFF);
      a.w = bf16_bits_to_float(w[1] >> 16);
      b.x = bf16_bits_to_float(w[2] & 0xFFFF);
      b.y = bf16_bits_to_float(w[2] >> 16);
      b.z = bf16_bits_to_float(w[3] & 0xFFFF);
      b.w = bf16_bits_to_float(w[3] >> 16);
      *reinterpret_cast<float4*>(dst + c * 8) = a;
      *reinterpret_cast<float4*>(dst + c * 8 + 4) = b;
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1) mla_decode_cuda_core_kernel(DecodeParams p) {
  extern __shared__ __align__(16) float smem[];
  float* sQ = smem;                          // [32][kStride]
  float* sK = sQ + kSubRows * kStride;       // [32][kStride]
  float* sP = sK + kTile * kStride;          // [32][kTile + 1]
  __shared__ int s_item, s_flag;
  __shared__ int s_valid[kTile];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  grid_dependency_wait();
  allow_dependent_launch();
  if (blockIdx.x == 0 && tid == 0) p.ws_hdr[kWsCounterWords] = p.counters_words;
  if (!plan_header_ok(p.plan, p)) {
    if (blockIdx.x == 0 && tid == 0) record_error(p.ws_hdr, MLA_DEV_PLAN_MISMATCH, 0);
    return;
  }
  const int n_items = p.plan[kHNItems];
  const int rr = tid >> 3;        // row within the 32-row pass
  const int cl = tid & 7;         // lane within the row's 8 threads

  for (;;) {
    __syncthreads();
    if (tid == 0) s_item = atomicAdd(&p.ws_hdr[kWsQueue], 1);
    __syncthreads();
    const int idx = s_item;
    if (idx >= n_items) break;
    const Item it = load_item(p, idx);
    if (!it.ok) continue;

    for (int sub = 0; sub < it.nrows; sub += kSubRows) {
      const int nsub = min(kSubRows, it.nrows - sub);
      __syncthreads();
      // Q rows of this pass -> fp32 shared memory (rows past nsub are zero).
      for (int r = warp; r < kSubRows; r += kThreads / 32) {
        float* dst = sQ + r * kStride;
        if (r < nsub) {
          const uint4* src = reinterpret_cast<const uint4*>(
              static_cast<const uint16_t*>(p.q) + (it.q_row_base + it.row0 + sub + r) * kDqk);
          for (int c = lane; c < kDqk / 8; c += 32) {
            const uint4 u = __ldg(src + c);
            const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              dst[c * 8 + 2 * k] = bf16_bits_to_float(w[k] & 0xFFFF);
              dst[c * 8 + 2 * k + 1] = bf16_bits_to_float(w[k] >> 16);
            }
          }
        } else {
          for (int c = lane; c < kDqk; c += 32) dst[c] = 0.f;
        }
      }
      const bool row_live = rr < nsub;
      const int t_row = row_live ? (it.row0 + sub + rr) / p.num_heads : 0;
      float m = -INFINITY, l = 0.f;
      float4 acc[16];
#pragma unroll
      for (int k = 0; k < 16; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);

      for (int e = it.e0; e < it.e1; e += kTile) {
        __syncthreads();
        // KV tile: warp w loads entries 4w .. 4w+3.
        for (int c = warp; c < kTile; c += kThreads / 32) {
          const int i = e + c;
          int ok = 0;
          int64_t slot = 0;
          if (i < it.e1) {
            const int32_t s = __ldg(p.kv_indices + it.kv_off + i);
            if (s >= 0 && s < p.num_slots) {
              ok = 1;
              slot = s;
            } else if (lane == 0) {
              record_error(p.ws_hdr, MLA_DEV_BAD_INDEX, (int)(it.kv_off + i));
            }
          }
          float* dst = sK + c * kStride;
          if (ok) {
            load_row_f32(p, slot, dst, lane);
          } else {
            for (int d = lane; d < kDqk; d += 32) dst[d] = 0.f;
          }
          if (lane == 0) s_valid[c] = ok;
        }
        __syncthreads();

        // S = Q K^T for row rr, entries cl + 8j.
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        const float* qrow = sQ + rr * kStride;
        for (int d = 0; d < kDqk; d += 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(qrow + d);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float4 k4 = *reinterpret_cast<const float4*>(sK + (cl + 8 * j) * kStride + d);
            sc[j] += q4.x * k4.x + q4.y * k4.y + q4.z * k4.z + q4.w * k4.w;
          }
        }
        float tmax = -INFINITY;
        bool vis[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int c = cl + 8 * j;
          vis[j] = row_live && s_valid[c] && visible(it, p, (int64_t)(e + c), t_row);
          sc[j] *= p.scale_log2;
          if (vis[j]) tmax = fmaxf(tmax, sc[j]);
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
        const float m_new = fmaxf(m, tmax);
        float alpha = 1.f, psum = 0.f;
        if (m_new != -INFINITY) {
          alpha = exp2f(m - m_new);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float pj = vis[j] ? exp2f(sc[j] - m_new) : 0.f;
            sP[rr * (kTile + 1) + cl + 8 * j] = pj;
            psum += pj;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) sP[rr * (kTile + 1) + cl + 8 * j] = 0.f;
        }
#pragma unroll
        for (int off = 1; off < 8; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
        l = l * alpha + psum;
        m = m_new;
        __syncthreads();

        // O = O * alpha + P V for row rr, dims 4*cl + 32k.
#pragma unroll
        for (int k = 0; k < 16; ++k) {
          acc[k].x *= alpha;
          acc[k].y *= alpha;
          acc[k].z *= alpha;
          acc[k].w *= alpha;
        }
        for (int c = 0; c < kTile; ++c) {
          const float pc = sP[rr * (kTile + 1) + c];
          const float* vrow = sK + c * kStride + 4 * cl;
#pragma unroll
          for (int k = 0; k < 16; ++k) {
            const float4 v4 = *reinterpret_cast<const float4*>(vrow + 32 * k);
            acc[k].x += pc * v4.x;
            acc[k].y += pc * v4.y;
            acc[k].z += pc * v4.z;
            acc[k].w += pc * v4.w;
          }
        }
      }

      // Epilogue of this pass.
      if (row_live) {
        const bool any = l > 0.f;
        const float inv = any ? p.out_scale / l : 0.f;
        const float lse = any ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
        const int rg = sub + rr;   // row within the group
        if (it.slot < 0) {
          const int64_t row = it.q_row_base + it.row0 + rg;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            store_o4(p, row, 4 * cl + 32 * k,
                     make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv));
          if (cl == 0) p.lse[row] = lse;
        } else {
          float* po = p.part_o + ((int64_t)it.slot * kRows + rg) * kDv;
#pragma unroll
          for (int k = 0; k < 16; ++k)
            *reinterpret_cast<float4*>(po + 4 * cl + 32 * k) =
                make_float4(acc[k].x * inv, acc[k].y * inv, acc[k].z * inv, acc[k].w * inv);
          if (cl == 0) p.part_lse[(int64_t)it.slot * kRows + rg] = lse;
        }
      }
    }
    if (it.slot >= 0) arrive_and_merge(p, it, &s_flag);
  }
  // The last worker out rewinds the queue for the next call: every worker's final
  // fetch is ordered before its count, and the count before the reset.
  if (tid == 0) {
    __threadfence();
    if (atomicAdd(&p.ws_hdr[kWsQueueDone], 1) == (int)gridDim.x - 1) {
      __threadfence();
      p.ws_hdr[kWsQueue] = 0;
      p.ws_hdr[kWsQueueDone] = 0;
    }
  }
}

}  // namespace

mla_status launch_decode_cuda_core(const DecodeParams& dp, void* stream) {
  const size_t smem = sizeof(float) * (size_t)(kSubRows * kStride + kTile * kStride + kSubRows * (kTile + 1));
  static bool attr_done[kMaxDevices] = {false};
  const int dev = current_device_slot();
  const int num_sms = device_sm_count(dev);
  if (num_sms == 0) return MLA_ERR_CUDA;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(mla_decode_cuda_core_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_done[dev] = true;
  }
  return launch_overlapped(mla_decode_cuda_core_kernel, dim3(num_sms), dim3(kThreads), smem, (cudaStream_t)stream,
                           dp) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace mla
