// pa_generic_bf16.cu -- instantiates the CUDA-core decode kernels for bf16
// elements (one translation unit per element type, compiled in parallel).
#include "pa_generic.cuh"

namespace pa {

cudaError_t launch_generic_bf16(const KernelArgs& a, bool v2, cudaStream_t s) {
  return launch_generic_dtype<__nv_bfloat16>(a, v2, s);
}

}  // namespace pa
