// pa_tc_f16.cu -- instantiates the tensor-core decode kernels for f16 caches
// (one translation unit per element type, compiled in parallel).
#include "pa_tc.cuh"

namespace pa {

cudaError_t launch_tc_f16(const KernelArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                         const CUtensorMap& qmap, const CUtensorMap& pmap, bool v2, int num_sms,
                         cudaStream_t s) {
  return launch_tc_dtype<__half>(a, kmap, vmap, qmap, pmap, v2, num_sms, s);
}

}  // namespace pa
