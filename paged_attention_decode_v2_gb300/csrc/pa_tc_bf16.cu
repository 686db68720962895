// pa_tc_bf16.cu -- instantiates the tensor-core decode kernels for bf16 caches
// (one translation unit per element type, compiled in parallel).
#include "pa_tc.cuh"

namespace pa {

cudaError_t launch_tc_bf16(const KernelArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const CUtensorMap& qmap, const CUtensorMap& pmap, bool v2, int num_sms,
                         cudaStream_t s) {
  return launch_tc_dtype<__nv_bfloat16>(a, kmap, vmap, qmap, pmap, v2, num_sms, s);
}

}  // namespace pa
