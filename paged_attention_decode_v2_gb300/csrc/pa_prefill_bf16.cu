// pa_prefill_bf16.cu -- bf16 instantiations of the tensor-core prefill kernel.
#include "pa_prefill.cuh"

namespace pa {

cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap (&m)[5], int num_sms,
                                cudaStream_t s) {
  return launch_prefill_dtype<__nv_bfloat16>(a, m, num_sms, s);
}

}  // namespace pa
