// pa_sx_f16.cu -- instantiates the split-x tensor-core decode kernels for f16
// caches (one translation unit per element type, compiled in parallel).
#include "pa_sx.cuh"

namespace pa {

cudaError_t launch_sx_f16(const KernelArgs& a, const CUtensorMap& pmap, bool v2, cudaStream_t s) {
  return launch_sx_dtype<__half>(a, pmap, v2, s);
}

}  // namespace pa
