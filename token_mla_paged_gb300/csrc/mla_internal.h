// Internal declarations shared by the host ABI layer and the CUDA kernels of
// the MLA paged-decode library.  Nothing here is part of the public ABI.
#pragma once

#include <utility>

#include <stddef.h>
#include <stdint.h>

#include "mla_gb300.h"

namespace mla {

constexpr int kDqk = MLA_D_QK;          // 576 = 512 latent + 64 RoPE
constexpr int kDv = MLA_D_V;            // 512
constexpr int kRows = MLA_ROWS_PER_GROUP;
constexpr int kBlockN = MLA_BLOCK_N;
constexpr int kMaxSplits = MLA_MAX_SPLITS;
constexpr int kMinTiles = 4;
constexpr int kCostClamp = 65535;

// ---------------------------------------------------------------- plan layout
// int32 words:  header[16] | S[B] | group_base[B+1] | partial_base[B] | items[cap][4]
constexpr int32_t kPlanMagic = 0x4D4C4150;
constexpr int32_t kPlanVersion = 1;
constexpr int kPlanHeaderInts = 16;
enum PlanHeader : int {
  kHMagic = 0, kHVersion, kHBatch, kHHeads, kHMaxQ, kHWorkers, kHMode, kHNItems, kHNPartials,
  kHNGroups, kHCapLo, kHCapHi, kHRows, kHBlockN, kHItemsCap, kHReserved
};

inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct PlanGeom {
  int32_t batch, g_max, items_cap;
  int64_t off_S, off_gbase, off_pbase, off_items, total_ints;
};

inline PlanGeom plan_geom(const mla_plan_params& p) {
  PlanGeom g;
  g.batch = p.batch;
  g.g_max = (int32_t)cdiv64((int64_t)p.num_heads * p.max_q_len, kRows);
  g.items_cap = (int32_t)((int64_t)p.num_workers + (int64_t)p.batch * g.g_max);
  g.off_S = kPlanHeaderInts;
  g.off_gbase = g.off_S + p.batch;
  g.off_pbase = g.off_gbase + p.batch + 1;
  g.off_items = g.off_pbase + p.batch;
  g.total_ints = g.off_items + 4LL * g.items_cap;
  return g;
}

// ---------------------------------------------------------------- workspace layout
// [0, 256)       header words: 0 error code, 1 error info (both persist until read),
//                2 queue head, 3 workers finished (CUDA-core kernel), 4 counter words
//                of the last call (written by the decode kernels)
// counters       int32 [2 * B * g_max]  split arrivals per (b, g, row half)
// The queue words and the counters start at zero (the workspace is zero-filled
// once, when it is allocated) and every call that completes leaves them at zero
// again: the last split of a group and the last worker to finish reset what they
// used.  A call that stopped on a device fault may leave them dirty, so reading the
// fault (mla_get_device_error) clears them.
// part_lse       fp32 [items_cap, 256]
// part_o         fp32 or bf16 [items_cap, 256, 512] (the tensor kernel stores bf16
//                partials when the output is bf16)
enum WsHeader : int { kWsErrCode = 0, kWsErrInfo = 1, kWsQueue = 2, kWsQueueDone = 3, kWsCounterWords = 4 };

struct WsGeom {
  size_t counters_off, part_lse_off, part_o_off, total;
  int64_t counters_cap, partial_cap;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline WsGeom ws_geom(const mla_plan_params& p) {
  PlanGeom pg = plan_geom(p);
  WsGeom w;
  w.counters_cap = 2 * (int64_t)p.batch * pg.g_max;
  if (w.counters_cap < 1) w.counters_cap = 1;
  w.partial_cap = pg.items_cap;
  w.counters_off = 256;
  w.part_lse_off = align_up(w.counters_off + 4 * (size_t)w.counters_cap, 256);
  w.part_o_off = align_up(w.part_lse_off + 4 * (size_t)w.partial_cap * kRows, 256);
  w.total = align_up(w.part_o_off + 4 * (size_t)w.partial_cap * kRows * kDv, 256);
  return w;
}

// ---------------------------------------------------------------- kernel params
struct DecodeParams {
  const void* q;
  const void* kv;
  int64_t num_slots;
  int32_t kv_fp8;
  int32_t out_fp32;
  const int32_t* kv_indptr;
  const int32_t* kv_indices;
  const int32_t* qo_indptr;
  const int32_t* pos_base_per_req;
  const int32_t* g_kv_indptr;
  int32_t causal, pos_base, pos_stride;
  const int32_t* kv_pos;  // nullable: per-entry global positions (ascending per request)
  int32_t window;         // sliding window on causal rows, 0 = none
  int32_t batch, num_heads, max_q_len, num_workers, mode, items_cap;
  float scale_log2;      // softmax_scale * kappa * log2(e): logits in base 2
  float out_scale;       // kappa (fp8) or 1: applied to the PV accumulator
  void* o;
  float* lse;
  const int32_t* plan;
  long long wait_limit;  // cycles a barrier wait may take before it reports MLA_DEV_WAIT_TIMEOUT
  int32_t test_stall;    // failure-path test: wait on a barrier nothing signals before any work
  int32_t* ws_hdr;
  int32_t* counters;     // split arrivals, [2 * B * g_max]
  int32_t counters_words;
  float* part_lse;
  float* part_o;
};

// ---------------------------------------------------------------- host planner
// Returns MLA_OK and fills `out` (plan_geom(p).total_ints words) or an error.
mla_status plan_build_host(const mla_plan_params& p, const int32_t* kv_indptr,
                           const int32_t* qo_indptr, int32_t* out);

// ---------------------------------------------------------------- launchers (.cu)
mla_status launch_plan_device(const mla_plan_params& p, const int32_t* kv_indptr,
                              const int32_t* qo_indptr, int32_t* plan, int32_t* ws_hdr,
                              void* stream);
// mla_decode_fwd; clear_state zeroes the queue words and split counters first
// (for a workspace that is not kept between calls).
mla_status decode_fwd_impl(const mla_fwd_args* a, void* stream, bool clear_state);
mla_status launch_decode_cuda_core(const DecodeParams& dp, void* stream);
mla_status launch_decode_tensor(const DecodeParams& dp, void* stream);
mla_status launch_merge_states(const void* o_parts, int o_parts_fp32, const float* lse_parts,
                               int n, int64_t rows, int dv, void* o, int o_fp32, float* lse,
                               void* stream);
mla_status launch_cache_write(const mla_cache_write_args& a, void* stream);
mla_status launch_rope_q_cache(const mla_rope_q_cache_args& a, void* stream);
mla_status launch_absorb_bmm(const mla_absorb_bmm_args& a, void* stream);
int tensor_kernel_available();
int tensor_kernel_workers();   // clusters of the tensor kernel resident at once (0 on error)

// Launch-time facts cached per device (opt-in shared-memory sizes, SM counts,
// occupancy): cudaFuncSetAttribute and the SM count belong to one device, so the
// launchers keep one entry per device index.  Returns the current device index,
// or -1 if it cannot be read or is >= kMaxDevices.  Two host threads that fill
// the same entry at once write the same values.
constexpr int kMaxDevices = 64;
int current_device_slot();
int device_sm_count(int dev);   // 0 on error

#ifdef __CUDACC__
// Programmatic dependent launch, device side: wait until the kernels this one may
// overlap have completed and their writes are visible (a no-op when it was
// launched in order), and let the next kernel on the stream start launching.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void allow_dependent_launch() { asm volatile("griddepcontrol.launch_dependents;" :::); }

// Launch with programmatic stream serialisation: the kernel may start while the
// kernel before it on the stream is still running, once every block of that
// kernel has signalled (griddepcontrol.launch_dependents) or exited.  The kernel
// must execute griddepcontrol.wait before it reads anything an earlier kernel
// wrote; the wait returns once the earlier kernels have completed and their
// writes are visible.  After a copy, a memset or a host node the launch is
// ordered as usual.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}
#endif

}  // namespace mla
