// tcgen05 bf16 varlen causal prefill (placeholder until the tensor-core kernel lands).
#include "astr_internal.cuh"
#include "launch.h"

namespace astr {

bool tc_prefill_supported(int, int, int, int) { return false; }

cudaError_t launch_tc_prefill(const astr_kv_cache &, int32_t, const void *, void *, int32_t,
                              uint64_t, uint32_t *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace astr
