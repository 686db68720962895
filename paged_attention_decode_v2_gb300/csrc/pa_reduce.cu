// pa_reduce.cu -- V2 pass 2: combine a row's partition results.
//
// For one (sequence b, query head h) with n = ceil(L / P) partitions, the
// pass-1 kernels left m_p (max logit), s_p (sum of exp(l - m_p)) and the
// normalised partial output o_p.  This kernel computes
//   M   = max_p m_p
//   w_p = exp(m_p - M) * s_p
//   out = sum_p w_p o_p / sum_p w_p
// which is the cross-partition log-sum-exp step of commit 4eb83a7e
// "qwen3_6_scripts", paragraph "Implementation (paged_attention_v2_pytorch
// .py)", Phase 2 (global_max, rescale, output), with total_sum read as the
// sum of the rescaled exp-sums.  Only partitions that exist are read, so the
// workspace needs no initialisation (the "shifted output" concern of the
// paragraph on test_device_scan_warpspeed_shifted_output, same page).
#include "pa_device.cuh"

namespace pa {

template <int D>
__global__ void __launch_bounds__(256) pa_reduce_kernel(const KernelArgs a) {
  constexpr int NT = 256, NW = NT / 32, E = D / 32;
  __shared__ float red[NW][D];
  __shared__ float wred[NW];
  __shared__ float smax[NW];
  __shared__ int snan[NW];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int h = blockIdx.x, b = blockIdx.y;
  const int64_t row = static_cast<int64_t>(b) * a.num_heads + h;

  // Wait for pass 1 (a no-op unless launched as a programmatic dependent).
  cudaGridDependencySynchronize();

  const int32_t L = a.seq_lens[b];
  if (!seq_len_ok(a, L) || L == 0) {
    const float v = L == 0 ? 0.f : qnan();
    for (int d = tid; d < D; d += NT) store_out(a.out, row * D + d, a.out_dtype, v);
    return;
  }
  const int n = (L + a.partition_size - 1) / a.partition_size;
  const float* __restrict__ ml = a.max_logits + row * a.num_partitions;
  const float* __restrict__ es = a.exp_sums + row * a.num_partitions;
  const float* __restrict__ to = a.tmp_out + row * a.num_partitions * D;

  // global max (and NaN detection: a pass-1 CTA that saw a bad block id
  // wrote NaN, which fmaxf would otherwise skip)
  float mx = -INFINITY;
  int has_nan = 0;
  for (int p = tid; p < n; p += NT) {
    const float v = ml[p];
    has_nan |= isnan(v);
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    has_nan |= __shfl_xor_sync(0xffffffffu, has_nan, o);
  }
  if (lane == 0) {
    smax[warp] = mx;
    snan[warp] = has_nan;
  }
  __syncthreads();
  float M = smax[0];
  int any_nan = snan[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) {
    M = fmaxf(M, smax[w]);
    any_nan |= snan[w];
  }

  // weighted sum: warp w takes partitions p = w, w + NW, ...; lanes split D
  float acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  float wsum = 0.f;
#pragma unroll 4
  for (int p = warp; p < n; p += NW) {
    const float w = es[p] * expf(ml[p] - M);
    float o[E];
    const float* src = to + static_cast<int64_t>(p) * D + lane * E;
#pragma unroll
    for (int e = 0; e < E; ++e) o[e] = src[e];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = fmaf(w, o[e], acc[e]);
    wsum += w;
  }
#pragma unroll
  for (int e = 0; e < E; ++e) red[warp][lane * E + e] = acc[e];
  if (lane == 0) wred[warp] = wsum;
  __syncthreads();
  float total = 0.f;
#pragma unroll
  for (int w = 0; w < NW; ++w) total += wred[w];
  for (int d = tid; d < D; d += NT) {
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) s += red[w][d];
    store_out(a.out, row * D + d, a.out_dtype, any_nan ? qnan() : s / total);
  }
}

template <int D>
static cudaError_t launch_reduce_d(const KernelArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(a.num_heads, a.num_seqs, 1);
  cfg.blockDim = dim3(256, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa_reduce_kernel<D>, a);
}

cudaError_t launch_reduce(const KernelArgs& a, cudaStream_t s, bool pdl) {
  switch (a.head_dim) {
    case 64: return launch_reduce_d<64>(a, s, pdl);
    case 128: return launch_reduce_d<128>(a, s, pdl);
    case 256: return launch_reduce_d<256>(a, s, pdl);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
