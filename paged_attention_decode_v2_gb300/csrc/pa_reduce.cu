// pa_reduce.cu -- V2 pass 2: combine a row's partition results.
//
// For one (sequence b, query head h) with n = ceil(L / P) partitions, pass 1
// left m_p (max logit), s_p (sum of exp(l - m_p)) and the normalised partial
// output o_p.  This kernel computes
//   M   = max_p m_p
//   w_p = exp(m_p - M) * s_p
//   out = sum_p w_p o_p / sum_p w_p
// which is the cross-partition log-sum-exp step of commit 4eb83a7e
// "qwen3_6_scripts", paragraph "Implementation (paged_attention_v2_pytorch
// .py)", Phase 2 (global_max, rescale, output), with total_sum read as the
// sum of the rescaled exp-sums.  Only partitions that exist are read, so the
// workspace needs no initialisation (the "shifted output" concern of the
// paragraph on test_device_scan_warpspeed_shifted_output, same page).
//
// Grid: (head_dim / 32, num_heads, num_seqs); each CTA produces 32 output
// elements of one row.  16 groups of 8 threads each fold a strided subset of
// the partitions into a running (max, weight, weighted sum) -- the same
// log-sum-exp identity applied incrementally -- and the groups are merged
// at the end.  Every load of a group is independent of the running values,
// so the partials are read with many loads in flight in one round.
#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kNT = 128;
constexpr int kSlice = 32;               // output elements per CTA
constexpr int kCols = kSlice / 4;        // float4 columns
constexpr int kGroups = kNT / kCols;     // partition groups

}  // namespace

template <int D>
__global__ void __launch_bounds__(kNT) pa_reduce_kernel(const KernelArgs a) {
  __shared__ float4 acc_s[kGroups][kCols];
  __shared__ float m_s[kGroups], w_s[kGroups];
  __shared__ int nan_s[kGroups];
  const int tid = threadIdx.x;
  const int x = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t row = static_cast<int64_t>(b) * a.num_heads + h;
  const int d0 = x * kSlice;

  // seq_lens is an input, not a pass-1 result: read it before waiting.
  const int32_t L = a.seq_lens[b];

  // Wait for pass 1 (a no-op unless launched as a programmatic dependent).
  cudaGridDependencySynchronize();

  if (!seq_len_ok(a, L) || L == 0) {
    const float v = L == 0 ? 0.f : qnan();
    if (tid < kSlice) store_out(a.out, row * D + d0 + tid, a.out_dtype, v);
    return;
  }
  const int n = (L + a.partition_size - 1) / a.partition_size;
  const float* __restrict__ ml = a.max_logits + row * a.num_partitions;
  const float* __restrict__ es = a.exp_sums + row * a.num_partitions;
  const float* __restrict__ to = a.tmp_out + row * a.num_partitions * D + d0;

  // Each group folds its partitions p = grp, grp + kGroups, ... into a
  // running (max, weight, weighted sum); all loads of a group are independent,
  // so a row of up to kGroups * 8 partitions is read in about one latency.
  const int col = tid % kCols, grp = tid / kCols;
  float m = -INFINITY, w = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int nan_seen = 0;
#pragma unroll 8
  for (int p = grp; p < n; p += kGroups) {
    const float mp = __ldg(ml + p);
    const float sp = __ldg(es + p);
    const float4 o = __ldg(reinterpret_cast<const float4*>(to + static_cast<int64_t>(p) * D) + col);
    nan_seen |= isnan(mp);
    if (mp > m) {
      const float f = expf(m - mp);  // 0 when m is -inf
      acc.x *= f;
      acc.y *= f;
      acc.z *= f;
      acc.w *= f;
      w *= f;
      m = mp;
    }
    const float e = sp * expf(mp - m);
    acc.x = fmaf(e, o.x, acc.x);
    acc.y = fmaf(e, o.y, acc.y);
    acc.z = fmaf(e, o.z, acc.z);
    acc.w = fmaf(e, o.w, acc.w);
    w += e;
  }
  acc_s[grp][col] = acc;
  if (col == 0) {
    m_s[grp] = m;
    w_s[grp] = w;
    nan_s[grp] = nan_seen;
  }
  __syncthreads();
  if (tid < kSlice) {
    float M = -INFINITY;
    int poison = 0;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      M = fmaxf(M, m_s[g]);
      poison |= nan_s[g];
    }
    float total = 0.f, s = 0.f;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const float f = m_s[g] == -INFINITY ? 0.f : expf(m_s[g] - M);
      total = fmaf(w_s[g], f, total);
      s = fmaf(reinterpret_cast<const float*>(&acc_s[g][tid / 4])[tid % 4], f, s);
    }
    store_out(a.out, row * D + d0 + tid, a.out_dtype, poison ? qnan() : s / total);
  }
}

template <int D>
static cudaError_t launch_reduce_d(const KernelArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(D / kSlice, a.num_heads, a.num_seqs);
  cfg.blockDim = dim3(kNT, 1, 1);
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
