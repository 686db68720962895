// pa_prefill_f16.cu -- f16 instantiations of the tensor-core prefill kernel.
#include "pa_prefill.cuh"

namespace pa {

cudaError_t launch_prefill_f16(const PrefillArgs& a, const CUtensorMap (&m)[5], int num_sms,
                               cudaStream_t s) {
  return launch_prefill_dtype<__half>(a, m, num_sms, s);
}

}  // namespace pa
