// pa_generic_f16.cu -- instantiates the CUDA-core decode kernels for f16
// elements (one translation unit per element type, compiled in parallel).
#include "pa_generic.cuh"

namespace pa {

cudaError_t launch_generic_f16(const KernelArgs& a, bool v2, cudaStream_t s) {
  return launch_generic_dtype<__half>(a, v2, s);
}

}  // namespace pa
