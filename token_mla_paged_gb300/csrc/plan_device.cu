// Device planner: rebuilds the work/split plan from the real per-request KV
// lengths at every call, so graph replays with growing KV get a split fitted
// to the lengths they actually have ("[DSV4] Tuned ASM FP8 decode with split
// plans; HCA on aiter's persistent V4-NM kernel", Summary part 2: the kernel
// plans the split from the real per-row KV lengths every call).
//
// One block of 64-1024 threads (sized to the batch and the item count: every
// block-wide barrier costs in proportion to the warps it waits for, and small
// problems are barrier-bound).  The output is bit-identical to the host planner
// on the same lengths: integer arithmetic only, and the cost-descending stable
// order is obtained by sorting unique keys ((65535 - cost) << 16 | enumeration
// index) with a bitonic network in shared memory.
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace mla {
namespace {

constexpr int kPlanThreadsMax = 1024;

// Exclusive scan of v[0..n) in place (int32), block-wide; returns the total.
__device__ int block_excl_scan(int* v, int n, int* warp_tmp) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nthreads = blockDim.x, nwarps = nthreads >> 5;
  const int per = (n + nthreads - 1) / nthreads;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int local = 0;
  for (int i = lo; i < hi; ++i) local += v[i];
  int incl = local;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += y;
  }
  if (lane == 31) warp_tmp[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? warp_tmp[lane] : 0;
    int wi = w;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, wi, off);
      if (lane >= off) wi += y;
    }
    warp_tmp[lane] = wi - w;        // exclusive prefix of warp totals
    if (lane == 31) warp_tmp[32] = wi;
  }
  __syncthreads();
  int run = warp_tmp[warp] + incl - local;
  for (int i = lo; i < hi; ++i) {
    const int x = v[i];
    v[i] = run;
    run += x;
  }
  const int total = warp_tmp[32];
  __syncthreads();
  return total;
}

__global__ void __launch_bounds__(kPlanThreadsMax, 1)
mla_plan_kernel(int B, int H, int max_q, int W, int items_cap, int p2cap,
                const int32_t* __restrict__ kv_indptr, const int32_t* __restrict__ qo_indptr,
                int32_t* __restrict__ plan, int32_t* __restrict__ ws_hdr) {
  extern __shared__ int sm[];
  int* sG = sm;                 // [B+1]
  int* sN = sG + (B + 1);       // [B+1]
  int* sS = sN + (B + 1);       // [B+1]
  int* sIb = sS + (B + 1);      // [B+1] item base (S*G scanned)
  int* sGb = sIb + (B + 1);     // [B+1] group base
  int* sPb = sGb + (B + 1);     // [B+1] partial base
  uint32_t* keys = reinterpret_cast<uint32_t*>(sPb + (B + 1));   // [p2cap]
  __shared__ int warp_tmp[33];
  __shared__ unsigned long long s_total;
  const int tid = threadIdx.x, nthreads = blockDim.x;
  // The lengths may come from the kernel before this one, and the plan buffer may
  // still be read by the previous call's decode: wait for both before touching them.
  grid_dependency_wait();
  allow_dependent_launch();   // the decode kernel's set-up may overlap this plan

  if (tid == 0) s_total = 0ull;
  __syncthreads();
  unsigned long long local_total = 0;
  for (int b = tid; b < B; b += nthreads) {
    int T = qo_indptr[b + 1] - qo_indptr[b];
    int L = kv_indptr[b + 1] - kv_indptr[b];
    if (T < 0 || L < 0) {
      record_error(ws_hdr, MLA_DEV_BAD_INDPTR, b);
      T = max(T, 0);
      L = max(L, 0);
    }
    if (T > max_q) {
      record_error(ws_hdr, MLA_DEV_ROWS_MISMATCH, b);
      T = max_q;
    }
    const int G = (int)(((int64_t)H * T + kRows - 1) / kRows);
    const int N = (int)(((int64_t)L + kBlockN - 1) / kBlockN);
    sG[b] = G;
    sN[b] = N;
    local_total += (unsigned long long)G * (unsigned long long)N;
  }
  atomicAdd(&s_total, local_total);
  __syncthreads();
  const int64_t total = (int64_t)s_total;
  int64_t target = (total + W - 1) / W;
  if (target < kMinTiles) target = kMinTiles;
  for (int b = tid; b < B; b += nthreads) {
    int64_t S = ((int64_t)sN[b] + target - 1) / target;
    S = S < 1 ? 1 : (S > kMaxSplits ? kMaxSplits : S);
    sS[b] = (int)S;
    sIb[b] = (int)S * sG[b];
    sGb[b] = sG[b];
    sPb[b] = S > 1 ? (int)S * sG[b] : 0;
  }
  __syncthreads();
  const int n_items_raw = block_excl_scan(sIb, B, warp_tmp);
  const int n_groups = block_excl_scan(sGb, B, warp_tmp);
  const int n_partials = block_excl_scan(sPb, B, warp_tmp);
  if (tid == 0) {
    sIb[B] = n_items_raw;
    sGb[B] = n_groups;
  }
  int n_items = n_items_raw;
  if (n_items > items_cap) {
    if (tid == 0) record_error(ws_hdr, MLA_DEV_PLAN_OVERFLOW, n_items_raw);
    n_items = items_cap;
  }
  __syncthreads();

  // Header and per-request arrays.
  const int64_t off_S = kPlanHeaderInts, off_g = off_S + B, off_p = off_g + B + 1,
                off_i = off_p + B;
  if (tid == 0) {
    plan[kHMagic] = kPlanMagic;
    plan[kHVersion] = kPlanVersion;
    plan[kHBatch] = B;
    plan[kHHeads] = H;
    plan[kHMaxQ] = max_q;
    plan[kHWorkers] = W;
    plan[kHMode] = MLA_PLAN_DYNAMIC;
    plan[kHNItems] = n_items;
    plan[kHNPartials] = n_partials;
    plan[kHNGroups] = n_groups;
    plan[kHCapLo] = 0;
    plan[kHCapHi] = 0;
    plan[kHRows] = kRows;
    plan[kHBlockN] = kBlockN;
    plan[kHItemsCap] = items_cap;
    plan[kHReserved] = 0;
  }
  for (int b = tid; b <= B; b += nthreads) {
    if (b < B) {
      plan[off_S + b] = sS[b];
      plan[off_p + b] = sS[b] > 1 ? sPb[b] : -1;
    }
    plan[off_g + b] = sGb[b];
  }

  // Sort keys: cost descending, then enumeration order.
  int p2 = 1;
  while (p2 < n_items) p2 <<= 1;
  for (int k = tid; k < p2; k += nthreads) keys[k] = 0xFFFFFFFFu;
  __syncthreads();
  for (int b = tid; b < B; b += nthreads) {
    const int S = sS[b], G = sG[b], N = sN[b];
    for (int s = 0; s < S; ++s) {
      const int64_t t0 = (int64_t)s * N / S, t1 = (int64_t)(s + 1) * N / S;
      const int64_t cost = (t1 - t0 + 1) < kCostClamp ? (t1 - t0 + 1) : (int64_t)kCostClamp;
      for (int g = 0; g < G; ++g) {
        const int e = sIb[b] + s * G + g;
        if (e < n_items) keys[e] = ((uint32_t)(kCostClamp - cost) << 16) | (uint32_t)e;
      }
    }
  }
  __syncthreads();
  for (int k = 2; k <= p2; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < p2; i += nthreads) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const uint32_t a = keys[i], c = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > c) == up) {
            keys[i] = c;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }
  for (int k = tid; k < items_cap; k += nthreads) {
    int32_t* rec = plan + off_i + 4LL * k;
    if (k < n_items) {
      const int e = (int)(keys[k] & 0xFFFFu);
      // request of enumeration index e: last b with item_base[b] <= e
      int lo = 0, hi = B;   // invariant: sIb[lo] <= e < sIb[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sIb[mid] <= e) lo = mid; else hi = mid;
      }
      const int b = lo, G = sG[b], q = e - sIb[b];
      rec[0] = b;
      rec[1] = q / G;
      rec[2] = q % G;
      rec[3] = sS[b] > 1 ? sPb[b] + q : -1;
    } else {
      rec[0] = rec[1] = rec[2] = rec[3] = 0;
    }
  }
}

}  // namespace

mla_status launch_plan_device(const mla_plan_params& p, const int32_t* kv_indptr,
                              const int32_t* qo_indptr, int32_t* plan, int32_t* ws_hdr,
                              void* stream) {
  const PlanGeom g = plan_geom(p);
  int p2cap = 1;
  while (p2cap < g.items_cap) p2cap <<= 1;
  const size_t smem = sizeof(int) * (6 * (size_t)(p.batch + 1) + (size_t)p2cap);
  static size_t attr_set[kMaxDevices] = {0};
  const int dev = current_device_slot();
  if (dev < 0) return MLA_ERR_CUDA;
  if (smem > 48 * 1024 && smem > attr_set[dev]) {
    if (cudaFuncSetAttribute(mla_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MLA_ERR_CUDA;
    attr_set[dev] = smem;
  }
  // threads: the larger of the batch and the item capacity, rounded up to a
  // power of two in [64, 1024]
  int threads = 64;
  while (threads < kPlanThreadsMax && (threads < p.batch + 1 || threads < g.items_cap)) threads <<= 1;
  return launch_overlapped(mla_plan_kernel, dim3(1), dim3(threads), smem, (cudaStream_t)stream, p.batch,
                           p.num_heads, p.max_q_len, p.num_workers, g.items_cap, p2cap, kv_indptr, qo_indptr,
                           plan, ws_hdr) == cudaSuccess
             ? MLA_OK
             : MLA_ERR_CUDA;
}

}  // namespace mla
