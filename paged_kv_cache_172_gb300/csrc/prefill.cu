// prefill.cu -- chunked prefill attention (tcgen05 tensor-core kernel).
// Placeholder until the tensor-core kernel lands: reports "unsupported".
#include "pk_common.cuh"
#include "pk_internal.h"

namespace pk {

bool prefill_supported(int, int) { return false; }

cudaError_t launch_prefill(const PrefillArgs&, const void*, const void*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace pk
