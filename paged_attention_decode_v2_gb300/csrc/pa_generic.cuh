// pa_generic.cuh -- CUDA-core decode kernels for every element type.
//
// One CTA handles one (sequence, KV head, token range).  The token range is
// one partition of partition_size tokens (V2 pass 1) or the whole sequence
// (V1).  The CTA serves all G query heads that share the KV head, so each
// key/value byte is read once per step no matter how many query heads use
// it (the grouped-query mapping of commit 4eb83a7e "qwen3_6_scripts",
// paragraph "V1 paged_attention (decode <= 8192)", head_mapping over 24
// query / 4 KV heads).
//
// The range is walked in chunks of CH tokens.  Per chunk:
//   1. the chunk's block ids are read from the block table (and checked);
//   2. QK^T: each warp takes U tokens at a time, lanes split head_dim, and
//      a butterfly reduce-scatter leaves one (token, head) logit per lane;
//   3. softmax statistics: warp h finds the chunk max of head h, turns the
//      logits into exp2(l - m) and folds the chunk into the running max and
//      sum (online rescaling across chunks, so V1 has no length limit);
//   4. P.V: each warp owns a head_dim slice, lanes split tokens, and the
//      partial sums are folded into the CTA's accumulator.
// Logits are kept in base-2 units (q is pre-multiplied by scale*log2(e)).
//
// These kernels are the portable path: they run for every dtype, head_dim
// and block size the ABI accepts, and they are the only path for float32.
// They also read the caches in the layout the same page gives for its V1
// kernel ("Hardware testing confirmed": keys [blocks, kv_heads, head_dim / x,
// block_size, x], values [blocks, kv_heads, head_dim, block_size]) when the
// call asks for it, x being the elements of one 16-byte group.
#pragma once

#include "pa_device.cuh"

namespace pa {

template <typename T, int D>
struct GenericCfg {
  static constexpr int NT = 256;              // threads per CTA
  static constexpr int NW = NT / 32;          // warps per CTA
  static constexpr int HP = 8;                // query heads per pass (== NW)
  static constexpr int CH = 256;              // tokens per chunk
  static constexpr int EPL = D / 32;          // QK: head_dim elements per lane
  static constexpr int U = 32 / HP;           // QK: tokens per warp step
  static constexpr int VEC = 16 / sizeof(T);  // PV: elements per 16-byte load
  static constexpr int X = 16 / sizeof(T);    // split-x layout: elements per key group
  static constexpr int KG = EPL < X ? EPL : X;  // QK: elements per contiguous key load
  static constexpr int WSLICE = D / NW;       // PV: head_dim slice per warp
  static constexpr int LPT = WSLICE / VEC;    // PV: lanes per token row
  static constexpr int TPS = 32 / LPT;        // PV: tokens per warp step
  static_assert(HP == NW, "one warp per head in the softmax step");
  static_assert(U * HP == 32, "reduce-scatter of 32 values");
  static_assert(LPT >= 1 && 32 % LPT == 0, "PV lane split");
};

template <int D>
struct GenericSmem {
  float q[8][D];     // scaled queries of the head group
  float acc[8][D];   // running sum_t exp2(l_t - m) V_t
  float p[256][8];   // chunk logits, then exp2(l - m)
  int32_t blk[258];  // chunk block ids (-1: outside the pool)
  float m_run[8];    // running max (base-2 units)
  float s_run[8];    // running sum of exp2(l - m_run)
  float factor[8];   // rescale of the accumulator for this chunk
  int bad;           // a block id of this range was outside the pool
};

// Butterfly reduce-scatter: on entry each lane holds 32 partial sums; on
// exit lane l returns the warp-wide total of value l.
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane) {
#pragma unroll
  for (int w = 16; w >= 1; w >>= 1) {
    const bool up = lane & w;
#pragma unroll
    for (int i = 0; i < w; ++i) {
      const float send = up ? v[i] : v[i + w];
      const float keep = up ? v[i + w] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, w);
    }
  }
  return v[0];
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

template <typename T, int D, bool kV2>
__global__ void __launch_bounds__(256) pa_generic_kernel(const KernelArgs a) {
  using C = GenericCfg<T, D>;
  __shared__ GenericSmem<D> sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b = blockIdx.z, kvh = blockIdx.y, part = blockIdx.x;
  const int BS = a.block_size, G = a.group, Hq = a.num_heads;
  const int32_t L = a.seq_lens[b];

  if (!seq_len_ok(a, L)) {
    if (tid == 0 && part == 0) set_status(a.status, PA_ERR_BAD_SEQ_LEN);
    if (!kV2) {  // V1 writes the NaN rows itself; the V2 reduce does it for V2
      for (int i = tid; i < G * D; i += C::NT)
        store_out(a.out, (static_cast<int64_t>(b) * Hq + kvh * G) * D + i, a.out_dtype, qnan());
    }
    return;
  }
  const int32_t t_begin = kV2 ? part * a.partition_size : 0;
  if (kV2 && t_begin >= L) return;  // this sequence has no such partition
  const int32_t t_end = kV2 ? min(L, t_begin + a.partition_size) : L;
  // a sequence that fits one partition is finished here (V1's contract)
  const bool direct = kV2 && a.single_direct && L <= a.partition_size;

  const T* __restrict__ kc = static_cast<const T*>(a.k_cache);
  const T* __restrict__ vc = static_cast<const T*>(a.v_cache);
  const T* __restrict__ qp = static_cast<const T*>(a.q);
  const int32_t* __restrict__ bt = a.block_tables + static_cast<int64_t>(b) * a.max_blocks_per_seq;
  const int64_t head_stride = static_cast<int64_t>(BS) * D;  // one (block, kv head) slice

  for (int hg = 0; hg * C::HP < G; ++hg) {
    const int nh = min(C::HP, G - hg * C::HP);
    const int h0 = kvh * G + hg * C::HP;  // first query head of this pass
    for (int i = tid; i < C::HP * D; i += C::NT) {
      const int hh = i / D, d = i % D;
      sm.q[hh][d] = hh < nh
          ? to_float(qp[(static_cast<int64_t>(b) * Hq + h0 + hh) * D + d]) * a.scale_log2
          : 0.f;
      sm.acc[hh][d] = 0.f;
    }
    if (tid < C::HP) {
      sm.m_run[tid] = -INFINITY;
      sm.s_run[tid] = 0.f;
    }
    if (tid == 0) sm.bad = 0;
    __syncthreads();

    for (int32_t c0 = t_begin; c0 < t_end; c0 += C::CH) {
      const int n = min(C::CH, t_end - c0);
      const int blk0 = c0 / BS;
      const int nblk = (c0 + n - 1) / BS - blk0 + 1;
      for (int j = tid; j < nblk; j += C::NT) {
        int32_t id = bt[blk0 + j];
        if (id < 0 || id >= a.num_blocks) {
          id = -1;
          sm.bad = 1;
          set_status(a.status, PA_ERR_BAD_BLOCK_ID);
        }
        sm.blk[j] = id;
      }
      __syncthreads();

      // ---- QK^T ------------------------------------------------------------
      for (int base = warp * C::U; base < n; base += C::NW * C::U) {
        float kf[C::U][C::EPL];
#pragma unroll
        for (int u = 0; u < C::U; ++u) {
          const int tt = base + u;
          const int t = c0 + tt;
          const int32_t id = tt < n ? sm.blk[t / BS - blk0] : -1;
          if (id >= 0) {
            const T* slice = kc + (static_cast<int64_t>(id) * a.num_kv_heads + kvh) * head_stride;
            if (!a.split_x) {
              load_row<T, C::EPL>(slice + static_cast<int64_t>(t % BS) * D + lane * C::EPL, kf[u]);
            } else {
              // element (slot s, d) at ((d / X) * BS + s) * X + d % X: this
              // lane's EPL elements are whole or part of 16-byte groups
#pragma unroll
              for (int g = 0; g < C::EPL / C::KG; ++g) {
                const int d = lane * C::EPL + g * C::KG;
                float f[C::KG];
                load_row<T, C::KG>(slice + (static_cast<int64_t>(d / C::X) * BS + t % BS) * C::X +
                                       d % C::X,
                                   f);
#pragma unroll
                for (int e = 0; e < C::KG; ++e) kf[u][g * C::KG + e] = f[e];
              }
            }
          } else {
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) kf[u][e] = 0.f;
          }
        }
        float part_sum[32];
#pragma unroll
        for (int h = 0; h < C::HP; ++h) {
          float qv[C::EPL];
#pragma unroll
          for (int e = 0; e < C::EPL; ++e) qv[e] = sm.q[h][lane * C::EPL + e];
#pragma unroll
          for (int u = 0; u < C::U; ++u) {
            float s = 0.f;
#pragma unroll
            for (int e = 0; e < C::EPL; ++e) s = fmaf(qv[e], kf[u][e], s);
            part_sum[u * C::HP + h] = s;
          }
        }
        const float logit = reduce_scatter32(part_sum, lane);
        const int tt = base + lane / C::HP;
        if (tt < n) {
          const int32_t id = sm.blk[(c0 + tt) / BS - blk0];
          sm.p[tt][lane % C::HP] = id >= 0 ? logit : -INFINITY;
        }
      }
      __syncthreads();

      // ---- softmax statistics: warp h owns head h ---------------------------
      {
        const int h = warp;
        float mx = -INFINITY;
        for (int tt = lane; tt < n; tt += 32) mx = fmaxf(mx, sm.p[tt][h]);
        mx = warp_max(mx);
        const float m_old = sm.m_run[h];
        const float m_new = fmaxf(m_old, mx);
        float sum = 0.f;
        for (int tt = lane; tt < n; tt += 32) {
          const float pv = m_new == -INFINITY ? 0.f : exp2f(sm.p[tt][h] - m_new);
          sm.p[tt][h] = pv;
          sum += pv;
        }
        sum = warp_sum(sum);
        if (lane == 0) {
          const float f = m_new == -INFINITY ? 1.f : exp2f(m_old - m_new);
          sm.factor[h] = f;
          sm.s_run[h] = sm.s_run[h] * f + sum;
          sm.m_run[h] = m_new;
        }
      }
      __syncthreads();

      // ---- P.V: warp owns head_dim slice, lanes split tokens ---------------
      {
        const int tl = lane / C::LPT, vi = lane % C::LPT;
        const int d0 = warp * C::WSLICE + vi * C::VEC;
        float acc[C::HP][C::VEC];
#pragma unroll
        for (int h = 0; h < C::HP; ++h)
#pragma unroll
          for (int e = 0; e < C::VEC; ++e) acc[h][e] = 0.f;
        for (int tt = tl; tt < n; tt += C::TPS) {
          const int t = c0 + tt;
          const int32_t id = sm.blk[t / BS - blk0];
          if (id < 0) continue;  // masked: never read its value row
          float vf[C::VEC];
          const T* vslice = vc + (static_cast<int64_t>(id) * a.num_kv_heads + kvh) * head_stride;
          if (!a.split_x) {
            load_row<T, C::VEC>(vslice + static_cast<int64_t>(t % BS) * D + d0, vf);
          } else {  // values [head_dim][block_size]: element (s, d) at d * BS + s
#pragma unroll
            for (int e = 0; e < C::VEC; ++e)
              vf[e] = to_float(vslice[static_cast<int64_t>(d0 + e) * BS + t % BS]);
          }
          const float4 pa4 = *reinterpret_cast<const float4*>(&sm.p[tt][0]);
          const float4 pb4 = *reinterpret_cast<const float4*>(&sm.p[tt][4]);
          const float pp[8] = {pa4.x, pa4.y, pa4.z, pa4.w, pb4.x, pb4.y, pb4.z, pb4.w};
#pragma unroll
          for (int h = 0; h < C::HP; ++h)
#pragma unroll
            for (int e = 0; e < C::VEC; ++e) acc[h][e] = fmaf(pp[h], vf[e], acc[h][e]);
        }
#pragma unroll
        for (int o = C::LPT; o < 32; o <<= 1)
#pragma unroll
          for (int h = 0; h < C::HP; ++h)
#pragma unroll
            for (int e = 0; e < C::VEC; ++e)
              acc[h][e] += __shfl_xor_sync(0xffffffffu, acc[h][e], o);
        if (tl == 0) {
#pragma unroll
          for (int h = 0; h < C::HP; ++h)
#pragma unroll
            for (int e = 0; e < C::VEC; ++e)
              sm.acc[h][d0 + e] = sm.acc[h][d0 + e] * sm.factor[h] + acc[h][e];
        }
      }
      __syncthreads();
    }

    // ---- epilogue ---------------------------------------------------------
    const bool bad = sm.bad != 0;
    for (int i = tid; i < nh * D; i += C::NT) {
      const int hh = i / D, d = i % D;
      const float s = sm.s_run[hh];
      const float o = bad ? qnan() : (s > 0.f ? sm.acc[hh][d] / s : 0.f);
      const int64_t row = static_cast<int64_t>(b) * Hq + h0 + hh;
      if (kV2 && !direct)
        a.tmp_out[(row * a.num_partitions + part) * D + d] = o;
      else
        store_out(a.out, row * D + d, a.out_dtype, o);
    }
    if (kV2 && !direct) {
      if (tid < nh) {
        const int64_t w = (static_cast<int64_t>(b) * Hq + h0 + tid) * a.num_partitions + part;
        a.max_logits[w] = bad ? qnan() : sm.m_run[tid] * kLn2;
        a.exp_sums[w] = sm.s_run[tid];
      }
    }
    __syncthreads();
  }
}

template <typename T, int D>
cudaError_t launch_generic_t(const KernelArgs& a, bool v2, cudaStream_t s) {
  const dim3 grid(v2 ? a.num_partitions : 1, a.num_kv_heads, a.num_seqs);
  if (v2)
    pa_generic_kernel<T, D, true><<<grid, GenericCfg<T, D>::NT, 0, s>>>(a);
  else
    pa_generic_kernel<T, D, false><<<grid, GenericCfg<T, D>::NT, 0, s>>>(a);
  return cudaGetLastError();
}

template <typename T>
cudaError_t launch_generic_dtype(const KernelArgs& a, bool v2, cudaStream_t s) {
  switch (a.head_dim) {
    case 64: return launch_generic_t<T, 64>(a, v2, s);
    case 128: return launch_generic_t<T, 128>(a, v2, s);
    case 256: return launch_generic_t<T, 256>(a, v2, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace pa
