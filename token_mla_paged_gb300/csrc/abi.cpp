// C ABI entry points: argument validation, plan/workspace sizing and kernel
// dispatch.  Every function returns a status and never aborts; nothing here
// allocates device memory, synchronises (except mla_get_device_error) or reads
// device memory on the host, so the forward path can be captured in a CUDA graph.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include <cuda_runtime.h>

#include "mla_internal.h"

using namespace mla;

namespace {

bool params_valid(const mla_plan_params* p) {
  if (!p) return false;
  if (p->batch < 0 || p->num_heads < 1 || p->max_q_len < 0 || p->num_workers < 1) return false;
  if (p->mode != MLA_PLAN_STATIC && p->mode != MLA_PLAN_DYNAMIC && p->mode != MLA_PLAN_HOST) return false;
  if (p->mode == MLA_PLAN_STATIC && p->kv_len_cap < 0) return false;
  return true;
}

bool aligned(const void* ptr, size_t a) { return ((uintptr_t)ptr % a) == 0; }

}  // namespace

namespace mla {

int current_device_slot() {
  int d = -1;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return -1;
  return d;
}

int device_sm_count(int dev) {
  static int sms[kMaxDevices] = {0};
  if (dev < 0 || dev >= kMaxDevices) return 0;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    sms[dev] = n;
  }
  return sms[dev];
}

mla_status decode_fwd_impl(const mla_fwd_args* a, void* stream, bool clear_state) {
  if (!a || !params_valid(a->params)) return MLA_ERR_INVALID_ARG;
  const mla_plan_params& p = *a->params;
  if (a->kv_dtype != MLA_KV_BF16 && a->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (a->out_dtype != MLA_OUT_BF16 && a->out_dtype != MLA_OUT_FP32) return MLA_ERR_INVALID_ARG;
  if (a->algo != MLA_ALGO_TENSOR && a->algo != MLA_ALGO_CUDA_CORE) return MLA_ERR_INVALID_ARG;
  if (a->causal != 0 && a->causal != 1) return MLA_ERR_INVALID_ARG;
  if (!(std::isfinite(a->softmax_scale) && a->softmax_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (a->kv_dtype == MLA_KV_FP8_E4M3 && !(std::isfinite(a->kv_scale) && a->kv_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (a->pos_stride < 1) return MLA_ERR_INVALID_ARG;
  if (a->window < 0 || (a->kv_pos && !aligned(a->kv_pos, 4))) return MLA_ERR_INVALID_ARG;
  if (a->num_slots <= 0 || a->num_slots > (int64_t)INT32_MAX) return MLA_ERR_INVALID_ARG;
  if (p.batch > 0) {
    if (!a->q || !a->kv_pool || !a->kv_indptr || !a->kv_indices || !a->qo_indptr || !a->o ||
        !a->lse)
      return MLA_ERR_INVALID_ARG;
    if (!aligned(a->q, 16) || !aligned(a->kv_pool, 16) || !aligned(a->o, 16) ||
        !aligned(a->lse, 4) || !aligned(a->kv_indptr, 4) || !aligned(a->kv_indices, 4) ||
        !aligned(a->qo_indptr, 4))
      return MLA_ERR_INVALID_ARG;
  }
  if (!a->plan_d || !a->workspace_d) return MLA_ERR_INVALID_ARG;
  if (!aligned(a->plan_d, 16) || !aligned(a->workspace_d, 256)) return MLA_ERR_INVALID_ARG;
  const PlanGeom pg = plan_geom(p);
  if (pg.items_cap > kCostClamp) return MLA_ERR_UNSUPPORTED;
  if (a->plan_bytes < sizeof(int32_t) * (size_t)pg.total_ints) return MLA_ERR_WORKSPACE_TOO_SMALL;
  const WsGeom wg = ws_geom(p);
  if (a->ws_bytes < wg.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (a->algo == MLA_ALGO_TENSOR && !tensor_kernel_available()) return MLA_ERR_UNSUPPORTED;
  if (p.mode == MLA_PLAN_DYNAMIC && (p.batch > 4096 || pg.items_cap > 8192))
    return MLA_ERR_UNSUPPORTED;

  char* ws = (char*)a->workspace_d;
  cudaStream_t st = (cudaStream_t)stream;
  // The queue words and split counters are left at zero by every completed call;
  // a caller whose workspace is not kept between calls asks for them to be cleared.
  if (clear_state &&
      cudaMemsetAsync(ws + 8, 0, wg.counters_off - 8 + 4 * (size_t)wg.counters_cap, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (p.batch == 0) return MLA_OK;
  if (p.mode == MLA_PLAN_DYNAMIC) {
    mla_status s = launch_plan_device(p, a->kv_indptr, a->qo_indptr, (int32_t*)a->plan_d,
                                      (int32_t*)ws, stream);
    if (s != MLA_OK) return s;
  }

  DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.q = a->q;
  dp.kv = a->kv_pool;
  dp.num_slots = a->num_slots;
  dp.kv_fp8 = a->kv_dtype == MLA_KV_FP8_E4M3;
  dp.out_fp32 = a->out_dtype == MLA_OUT_FP32;
  dp.kv_indptr = a->kv_indptr;
  dp.kv_indices = a->kv_indices;
  dp.qo_indptr = a->qo_indptr;
  dp.pos_base_per_req = a->pos_base_per_req;
  dp.g_kv_indptr = a->g_kv_indptr;
  dp.causal = a->causal;
  dp.pos_base = a->pos_base;
  dp.pos_stride = a->pos_stride;
  dp.kv_pos = a->kv_pos;
  dp.window = a->window;
  dp.batch = p.batch;
  dp.num_heads = p.num_heads;
  dp.max_q_len = p.max_q_len;
  dp.num_workers = p.num_workers;
  dp.mode = p.mode;
  dp.items_cap = pg.items_cap;
  const float kappa = dp.kv_fp8 ? a->kv_scale : 1.0f;
  dp.scale_log2 = (float)((double)a->softmax_scale * (double)kappa * 1.4426950408889634);
  dp.out_scale = kappa;
  dp.o = a->o;
  dp.lse = a->lse;
  dp.plan = (const int32_t*)a->plan_d;
  dp.wait_limit = 2000000000LL;   // about a second at GB300 clocks
  // Failure-path test hook (tests only): MLA_TEST_STALL_CYCLES=<n> makes the
  // tensor kernel wait on a barrier nothing signals, with a limit of n cycles.
  if (const char* e = std::getenv("MLA_TEST_STALL_CYCLES")) {
    const long long n = std::atoll(e);
    if (n > 0) {
      dp.test_stall = 1;
      dp.wait_limit = n;
    }
  }
  dp.ws_hdr = (int32_t*)ws;
  dp.counters = (int32_t*)(ws + wg.counters_off);
  dp.counters_words = (int32_t)wg.counters_cap;
  dp.part_lse = (float*)(ws + wg.part_lse_off);
  dp.part_o = (float*)(ws + wg.part_o_off);
  return a->algo == MLA_ALGO_TENSOR ? launch_decode_tensor(dp, stream)
                                    : launch_decode_cuda_core(dp, stream);
}

}  // namespace mla

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_status_string(int status) {
  switch (status) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "plan or workspace buffer too small";
    case MLA_ERR_PLAN_MISMATCH: return "plan does not match the call";
    case MLA_ERR_CUDA: return "CUDA runtime error";
    case MLA_ERR_DEVICE_FAULT: return "device-side fault recorded in the workspace";
    default: return "unknown status";
  }
}

mla_status mla_decode_workers(int32_t algo, int32_t* num_workers) {
  if (!num_workers || (algo != MLA_ALGO_TENSOR && algo != MLA_ALGO_CUDA_CORE)) return MLA_ERR_INVALID_ARG;
  const int n = algo == MLA_ALGO_TENSOR ? tensor_kernel_workers() : device_sm_count(current_device_slot());
  if (n < 1) return MLA_ERR_CUDA;
  *num_workers = n;
  return MLA_OK;
}

mla_status mla_decode_plan_size(const mla_plan_params* params, size_t* plan_bytes,
                                size_t* workspace_bytes) {
  if (!params_valid(params)) return MLA_ERR_INVALID_ARG;
  const PlanGeom pg = plan_geom(*params);
  if (pg.items_cap > kCostClamp) return MLA_ERR_UNSUPPORTED;
  if (plan_bytes) *plan_bytes = sizeof(int32_t) * (size_t)pg.total_ints;
  if (workspace_bytes) *workspace_bytes = ws_geom(*params).total;
  return MLA_OK;
}

mla_status mla_decode_plan(const mla_plan_params* params, const int32_t* kv_indptr_h,
                           const int32_t* qo_indptr_h, void* plan_h, size_t plan_bytes) {
  if (!params_valid(params) || !plan_h) return MLA_ERR_INVALID_ARG;
  const PlanGeom pg = plan_geom(*params);
  if (plan_bytes < sizeof(int32_t) * (size_t)pg.total_ints) return MLA_ERR_WORKSPACE_TOO_SMALL;
  return plan_build_host(*params, kv_indptr_h, qo_indptr_h, (int32_t*)plan_h);
}

mla_status mla_decode_plan_device(const mla_plan_params* params, const int32_t* kv_indptr_d,
                                  const int32_t* qo_indptr_d, void* plan_d, size_t plan_bytes,
                                  void* workspace_d, size_t ws_bytes, void* stream) {
  if (!params_valid(params) || !plan_d || !workspace_d) return MLA_ERR_INVALID_ARG;
  if (params->mode != MLA_PLAN_DYNAMIC) return MLA_ERR_INVALID_ARG;
  if (params->batch > 0 && (!kv_indptr_d || !qo_indptr_d)) return MLA_ERR_INVALID_ARG;
  const PlanGeom pg = plan_geom(*params);
  if (params->batch > 4096 || pg.items_cap > 8192) return MLA_ERR_UNSUPPORTED;
  if (plan_bytes < sizeof(int32_t) * (size_t)pg.total_ints) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (ws_bytes < ws_geom(*params).total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (!aligned(plan_d, 16) || !aligned(workspace_d, 256)) return MLA_ERR_INVALID_ARG;
  return launch_plan_device(*params, kv_indptr_d, qo_indptr_d, (int32_t*)plan_d,
                            (int32_t*)workspace_d, stream);
}

mla_status mla_decode_fwd(const mla_fwd_args* a, void* stream) {
  return decode_fwd_impl(a, stream, false);
}

mla_status mla_merge_states(const void* o_parts, int32_t o_parts_dtype, const float* lse_parts,
                            int32_t n, int64_t rows, int32_t dv, void* o, int32_t o_dtype,
                            float* lse, void* stream) {
  if (n < 1 || rows < 0 || dv < 1) return MLA_ERR_INVALID_ARG;
  if (o_parts_dtype != MLA_OUT_BF16 && o_parts_dtype != MLA_OUT_FP32) return MLA_ERR_INVALID_ARG;
  if (o_dtype != MLA_OUT_BF16 && o_dtype != MLA_OUT_FP32) return MLA_ERR_INVALID_ARG;
  if (rows == 0) return MLA_OK;
  if (!o_parts || !lse_parts || !o || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(o_parts, 4) || !aligned(lse_parts, 4) || !aligned(o, 4) || !aligned(lse, 4))
    return MLA_ERR_INVALID_ARG;
  return launch_merge_states(o_parts, o_parts_dtype == MLA_OUT_FP32, lse_parts, n, rows, dv, o,
                             o_dtype == MLA_OUT_FP32, lse, stream);
}

mla_status mla_cache_write(const mla_cache_write_args* a, void* stream) {
  if (!a) return MLA_ERR_INVALID_ARG;
  if (a->kv_c_dtype != MLA_ACT_BF16 && a->kv_c_dtype != MLA_ACT_FP32) return MLA_ERR_INVALID_ARG;
  if (a->k_pe_dtype != MLA_ACT_BF16 && a->k_pe_dtype != MLA_ACT_FP32) return MLA_ERR_INVALID_ARG;
  if (a->kv_dtype != MLA_KV_BF16 && a->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->num_slots <= 0) return MLA_ERR_INVALID_ARG;
  if (a->kv_c_stride < 512 || a->k_pe_stride < 64) return MLA_ERR_INVALID_ARG;
  if (a->kv_dtype == MLA_KV_FP8_E4M3 && !(std::isfinite(a->kv_scale) && a->kv_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (a->num_tokens == 0) return MLA_OK;
  if (!a->kv_c || !a->k_pe || !a->slot_mapping || !a->kv_pool) return MLA_ERR_INVALID_ARG;
  // 16-byte rows: aligned bases, strides a whole number of 16-byte units
  const int64_t c_unit = a->kv_c_dtype == MLA_ACT_FP32 ? 4 : 8, pe_unit = a->k_pe_dtype == MLA_ACT_FP32 ? 4 : 8;
  if (!aligned(a->kv_c, 16) || !aligned(a->k_pe, 16) || !aligned(a->kv_pool, 16) || !aligned(a->slot_mapping, 4) ||
      a->kv_c_stride % c_unit != 0 || a->k_pe_stride % pe_unit != 0)
    return MLA_ERR_INVALID_ARG;
  return launch_cache_write(*a, stream);
}

mla_status mla_rope_q_cache(const mla_rope_q_cache_args* a, void* stream) {
  if (!a) return MLA_ERR_INVALID_ARG;
  if (a->num_heads < 1 || a->num_tokens < 0 || a->max_pos < 1 || a->num_slots <= 0) return MLA_ERR_INVALID_ARG;
  if (a->rope_style != MLA_ROPE_NEOX && a->rope_style != MLA_ROPE_INTERLEAVED) return MLA_ERR_INVALID_ARG;
  if (a->kv_dtype != MLA_KV_BF16 && a->kv_dtype != MLA_KV_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (a->kv_dtype == MLA_KV_FP8_E4M3 && !(std::isfinite(a->kv_scale) && a->kv_scale > 0.f))
    return MLA_ERR_INVALID_ARG;
  if (a->kv_c_stride < 512 || a->k_pe_stride < 64) return MLA_ERR_INVALID_ARG;
  if (a->num_tokens == 0) return MLA_OK;
  if (!a->q_nope || !a->q_pe || !a->q_out || !a->kv_c || !a->k_pe || !a->positions || !a->cos_sin ||
      !a->slot_mapping || !a->kv_pool)
    return MLA_ERR_INVALID_ARG;
  const int64_t strides[] = {a->q_nope_stride_token, a->q_nope_stride_head, a->q_pe_stride_token,
                             a->q_pe_stride_head, a->kv_c_stride, a->k_pe_stride};
  for (int64_t st : strides)
    if (st < 0 || st % 8 != 0) return MLA_ERR_INVALID_ARG;
  if (!aligned(a->q_nope, 16) || !aligned(a->q_pe, 16) || !aligned(a->q_out, 16) || !aligned(a->kv_c, 16) ||
      !aligned(a->k_pe, 16) || !aligned(a->kv_pool, 16) || !aligned(a->cos_sin, 4) ||
      !aligned(a->positions, 4) || !aligned(a->slot_mapping, 4))
    return MLA_ERR_INVALID_ARG;
  return launch_rope_q_cache(*a, stream);
}

mla_status mla_absorb_bmm(const mla_absorb_bmm_args* a, void* stream) {
  if (!a) return MLA_ERR_INVALID_ARG;
  if (a->num_tokens < 0 || a->num_heads < 1 || a->num_heads > 65535) return MLA_ERR_INVALID_ARG;
  if (a->k < 64 || a->k > 8192 || a->k % 64 != 0 || a->n < 128 || a->n > 8192 || a->n % 128 != 0)
    return MLA_ERR_INVALID_ARG;
  if (a->w_dtype != MLA_W_BF16 && a->w_dtype != MLA_W_FP8_E4M3) return MLA_ERR_INVALID_ARG;
  if (!std::isfinite(a->w_scale)) return MLA_ERR_INVALID_ARG;
  if (a->x_stride_head < a->k || a->out_stride_head < a->n || a->x_stride_token < 0 || a->out_stride_token < 0)
    return MLA_ERR_INVALID_ARG;
  const int64_t strides[] = {a->x_stride_token, a->x_stride_head, a->out_stride_token, a->out_stride_head};
  for (int64_t st : strides)
    if (st % 8 != 0) return MLA_ERR_INVALID_ARG;
  if (a->num_tokens == 0) return MLA_OK;
  if (!a->x || !a->w || !a->out) return MLA_ERR_INVALID_ARG;
  if (!aligned(a->x, 16) || !aligned(a->w, 16) || !aligned(a->out, 16) || !aligned(a->status_d, 4))
    return MLA_ERR_INVALID_ARG;
  return launch_absorb_bmm(*a, stream);
}

mla_status mla_get_device_error(void* workspace_d, void* stream, int32_t* code, int32_t* info) {
  if (!workspace_d || !code) return MLA_ERR_INVALID_ARG;
  int32_t h[kWsCounterWords + 1] = {0};
  cudaStream_t st = (cudaStream_t)stream;
  if (cudaMemcpyAsync(h, workspace_d, sizeof(h), cudaMemcpyDeviceToHost, st) != cudaSuccess)
    return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  // A call that stopped on a fault may have left the queue words or split
  // counters (header word 4 holds how many the last call used) non-zero.
  const size_t clear = h[0] == 0 ? 2 * sizeof(int32_t)
                                 : 256 + sizeof(int32_t) * (size_t)(h[kWsCounterWords] > 0 ? h[kWsCounterWords] : 0);
  if (cudaMemsetAsync(workspace_d, 0, clear, st) != cudaSuccess) return MLA_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return MLA_ERR_CUDA;
  *code = h[0];
  if (info) *info = h[1];
  return h[0] == 0 ? MLA_OK : MLA_ERR_DEVICE_FAULT;
}

}  // extern "C"
