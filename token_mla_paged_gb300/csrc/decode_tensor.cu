// Tensor-core (tcgen05 / TMEM) MLA decode kernel for sm_103a.
#include <cuda_runtime.h>

#include "device_common.cuh"

namespace mla {

int tensor_kernel_available() { return 0; }

mla_status launch_decode_tensor(const DecodeParams&, void*) { return MLA_ERR_UNSUPPORTED; }

}  // namespace mla
