// Forward entry point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a custom allocator that owns every
// byte of the device, an inference runtime that hands out only the input and
// output tensors, or code that runs inside a context where allocation is not
// allowed.  They still need the decode, which needs a plan buffer and a
// workspace (split partials, merge counters, queue heads, error word).  This
// entry point takes that scratch from one file-scope device array instead.
//
// The array is kNoAllocScratchBytes (16 MiB) and lives as long as the library
// is loaded on a device: every GPU that loads the library holds it until the
// process exits.  Its device address is looked up once per device, on the first
// call made with that device current (cudaGetSymbolAddress); make that first
// call before any stream capture.  The address is kept in an atomic slot: host
// threads whose first calls coincide each look it up and store the same value.
// All calls share the array and it keeps the
// last call's contents, so two calls that overlap on the GPU (different streams
// without ordering) race on it.  What must start at zero is cleared by every
// call (queue heads and split-merge counters); the plan is rebuilt on the device
// by every call, which is why only the re-planning (DYNAMIC) mode is accepted.
#include <atomic>

#include <cuda_runtime.h>

#include "mla_internal.h"

namespace mla {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::atomic<void*> g_scratch_addr[kMaxDevices];   // zero-initialised (static storage)

}  // namespace
}  // namespace mla

using namespace mla;

extern "C" mla_status mla_decode_fwd_noalloc(const mla_fwd_args* args, void* stream) {
  if (!args || !args->params) return MLA_ERR_INVALID_ARG;
  const mla_plan_params& p = *args->params;
  if (p.mode != MLA_PLAN_DYNAMIC) return MLA_ERR_UNSUPPORTED;
  size_t plan_bytes = 0, ws_bytes = 0;
  const mla_status s = mla_decode_plan_size(&p, &plan_bytes, &ws_bytes);
  if (s != MLA_OK) return s;
  const size_t plan_span = align_up(plan_bytes, 256);
  if (plan_span + ws_bytes > kNoAllocScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  void* base = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (base == nullptr) {
    // Host code must not use the array's name as an address: ask the runtime for
    // the device address of this device's copy.
    if (cudaGetSymbolAddress(&base, g_noalloc_scratch) != cudaSuccess || base == nullptr) return MLA_ERR_CUDA;
    g_scratch_addr[dev].store(base, std::memory_order_release);
  }
  mla_fwd_args a = *args;
  a.plan_d = base;
  a.plan_bytes = plan_bytes;
  a.workspace_d = static_cast<unsigned char*>(base) + plan_span;
  a.ws_bytes = kNoAllocScratchBytes - plan_span;
  return decode_fwd_impl(&a, stream, true);
}
