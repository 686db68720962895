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
// Grid: (head_dim / S, num_heads, num_seqs); each CTA of 128 threads
// produces S output elements of one row (S = 32, 64, 128 or 256, chosen per
// launch so that large batches do not need many waves of tiny CTAs).  The
// threads form 512 / S groups of S / 4 threads (one float4 column each);
// group g folds partitions g, g + groups, ... into a running (max, weight,
// weighted sum) -- the same log-sum-exp identity applied incrementally --
// and the groups are merged at the end.  A thread loads a batch of its
// partitions at once (statistics and partial output, all independent of the
// running values) before it folds them, so a row is read in
// ceil(n / (groups * batch)) rounds of memory latency (batches of 4, with
// at most 64 registers a thread: eight CTAs resident per SM).
#include "pa_device.cuh"

namespace pa {

namespace {

constexpr int kNT = 128;

// Partitions a thread has in flight, and the CTAs per SM the register
// budget is set for.  Few registers matter more than many loads in flight:
// reduce CTAs that fit beside pass 1's CTAs on an SM are resident (waiting
// on the grid dependency) before pass 1 ends.  Measured on GB300 over
// batches of 4 / 8 / 16 loads with 4-8 CTAs per SM: 4 loads and at most 64
// registers was the fastest on every workload.
constexpr int kBatch = 4;
constexpr int kMinBlocks = 8;

}  // namespace

template <int D, int S>
__global__ void __launch_bounds__(kNT, kMinBlocks) pa_reduce_kernel(const KernelArgs a) {
  constexpr int kCols = S / 4;           // float4 columns of the slice
  constexpr int kGroups = kNT / kCols;   // partition groups
  static_assert(kGroups >= 1 && kCols * kGroups == kNT, "slice width");
  __shared__ float4 acc_s[kGroups][kCols];
  __shared__ float m_s[kGroups], w_s[kGroups];
  __shared__ int nan_s[kGroups];
  const int tid = threadIdx.x;
  const int x = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int64_t row = static_cast<int64_t>(b) * a.num_heads + h;
  const int d0 = x * S;

  // seq_lens is an input, not a pass-1 result: read it before waiting.
  const int32_t L = a.seq_lens[b];
  // a sequence of one partition was finished by pass 1 (single_direct)
  if (a.single_direct && L >= 1 && L <= a.partition_size && seq_len_ok(a, L)) return;

  // Wait for pass 1 (a no-op unless launched as a programmatic dependent).
  cudaGridDependencySynchronize();

  if (!seq_len_ok(a, L) || L == 0) {
    const float v = L == 0 ? 0.f : qnan();
    for (int c = tid; c < kCols; c += kNT)
      store_out4(a.out, row * D + d0 + 4 * c, a.out_dtype, make_float4(v, v, v, v));
    return;
  }
  const int n = (L + a.partition_size - 1) / a.partition_size;
  const float* __restrict__ ml = a.max_logits + row * a.num_partitions;
  const float* __restrict__ es = a.exp_sums + row * a.num_partitions;
  const float4* __restrict__ to =
      reinterpret_cast<const float4*>(a.tmp_out + row * a.num_partitions * D + d0);

  const int col = tid % kCols, grp = tid / kCols;
  float m = -INFINITY, w = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  int nan_seen = 0;
  for (int base = grp; base < n; base += kGroups * kBatch) {
    float mp[kBatch], sp[kBatch];
    float4 o[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      const int p = base + i * kGroups;
      if (p < n) {
        mp[i] = __ldg(ml + p);
        sp[i] = __ldg(es + p);
        o[i] = __ldg(to + static_cast<int64_t>(p) * (D / 4) + col);
      } else {
        mp[i] = -INFINITY;
        sp[i] = 0.f;
        o[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    // the batch's max moves the running reference once
    float mb = m;
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      nan_seen |= isnan(mp[i]);
      mb = fmaxf(mb, mp[i]);
    }
    if (mb > m) {
      const float f = expf(m - mb);  // 0 when m is -inf
      acc.x *= f;
      acc.y *= f;
      acc.z *= f;
      acc.w *= f;
      w *= f;
      m = mb;
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i) {
      if (base + i * kGroups < n) {
        const float e = sp[i] * expf(mp[i] - m);
        acc.x = fmaf(e, o[i].x, acc.x);
        acc.y = fmaf(e, o[i].y, acc.y);
        acc.z = fmaf(e, o[i].z, acc.z);
        acc.w = fmaf(e, o[i].w, acc.w);
        w += e;
      }
    }
  }
  acc_s[grp][col] = acc;
  if (col == 0) {
    m_s[grp] = m;
    w_s[grp] = w;
    nan_s[grp] = nan_seen;
  }
  __syncthreads();
  for (int c = tid; c < kCols; c += kNT) {
    float M = -INFINITY;
    int poison = 0;
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      M = fmaxf(M, m_s[g]);
      poison |= nan_s[g];
    }
    float total = 0.f;
    float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int g = 0; g < kGroups; ++g) {
      const float f = m_s[g] == -INFINITY ? 0.f : expf(m_s[g] - M);
      const float4 v = acc_s[g][c];
      total = fmaf(w_s[g], f, total);
      s.x = fmaf(v.x, f, s.x);
      s.y = fmaf(v.y, f, s.y);
      s.z = fmaf(v.z, f, s.z);
      s.w = fmaf(v.w, f, s.w);
    }
    const float4 r = poison ? make_float4(qnan(), qnan(), qnan(), qnan())
                            : make_float4(s.x / total, s.y / total, s.z / total, s.w / total);
    store_out4(a.out, row * D + d0 + 4 * c, a.out_dtype, r);
  }
}

template <int D, int S>
static cudaError_t launch_reduce_ds(const KernelArgs& a, cudaStream_t s, bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(D / S, a.num_heads, a.num_seqs);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, pa_reduce_kernel<D, S>, a);
}

// Output elements per CTA: 32 (the most groups per row, for long rows of
// small batches) unless that would take more than two waves of CTAs, in
// which case the slice widens (fewer, fuller CTAs) up to the whole row.
static int slice_width(const KernelArgs& a) {
  int sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      sms <= 0)
    sms = 148;
  const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.num_heads;
  int S = 32;
  while (S < a.head_dim && rows * (a.head_dim / S) > 2LL * sms * kMinBlocks) S *= 2;
  return S;
}

template <int D>
static cudaError_t launch_reduce_d(const KernelArgs& a, cudaStream_t s, bool pdl) {
  switch (slice_width(a)) {
    case 32: return launch_reduce_ds<D, 32>(a, s, pdl);
    case 64: return launch_reduce_ds<D, 64>(a, s, pdl);
    case 128:
      if constexpr (D >= 128) return launch_reduce_ds<D, 128>(a, s, pdl);
      break;
    case 256:
      if constexpr (D >= 256) return launch_reduce_ds<D, 256>(a, s, pdl);
      break;
  }
  return cudaErrorInvalidValue;
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
