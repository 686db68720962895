// pa_device.cuh -- small device helpers shared by the kernels: exact
// widening of bf16 / f16 / f32 elements to float, vector loads of KV rows,
// output stores and the device status word.
#pragma once

#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "pa_internal.h"

namespace pa {

constexpr float kLn2 = 0.693147180559945309417f;
constexpr float kLog2e = 1.442695040888963407360f;

// ---- exact widening of packed elements to float ---------------------------

// Two bf16 in one 32-bit word: a bf16 is the upper half of a binary32.
__device__ __forceinline__ void widen2(const __nv_bfloat16*, uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}
__device__ __forceinline__ void widen2(const __half*, uint32_t w, float& lo, float& hi) {
  __half2 h = *reinterpret_cast<__half2*>(&w);
  float2 f = __half22float2(h);
  lo = f.x;
  hi = f.y;
}

// Load N consecutive elements starting at p (aligned to N*sizeof(T), at most
// 32 bytes) and widen them to float.
template <typename T, int N>
__device__ __forceinline__ void load_row(const T* __restrict__ p, float (&f)[N]) {
  if constexpr (sizeof(T) == 4) {
    static_assert(N == 2 || N % 4 == 0, "f32 row slice");
    if constexpr (N == 2) {
      float2 v = __ldg(reinterpret_cast<const float2*>(p));
      f[0] = v.x;
      f[1] = v.y;
    } else {
#pragma unroll
      for (int i = 0; i < N / 4; ++i) {
        float4 v = __ldg(reinterpret_cast<const float4*>(p) + i);
        f[4 * i + 0] = v.x;
        f[4 * i + 1] = v.y;
        f[4 * i + 2] = v.z;
        f[4 * i + 3] = v.w;
      }
    }
  } else {
    static_assert(N == 2 || N == 4 || N % 8 == 0, "16-bit row slice");
    if constexpr (N == 2) {
      uint32_t w = __ldg(reinterpret_cast<const unsigned int*>(p));
      widen2(p, w, f[0], f[1]);
    } else if constexpr (N == 4) {
      uint2 w = __ldg(reinterpret_cast<const uint2*>(p));
      widen2(p, w.x, f[0], f[1]);
      widen2(p, w.y, f[2], f[3]);
    } else {
#pragma unroll
      for (int i = 0; i < N / 8; ++i) {
        uint4 w = __ldg(reinterpret_cast<const uint4*>(p) + i);
        widen2(p, w.x, f[8 * i + 0], f[8 * i + 1]);
        widen2(p, w.y, f[8 * i + 2], f[8 * i + 3]);
        widen2(p, w.z, f[8 * i + 4], f[8 * i + 5]);
        widen2(p, w.w, f[8 * i + 6], f[8 * i + 7]);
      }
    }
  }
}

__device__ __forceinline__ float to_float(float x) { return x; }
__device__ __forceinline__ float to_float(__nv_bfloat16 x) { return __bfloat162float(x); }
__device__ __forceinline__ float to_float(__half x) { return __half2float(x); }

// Store one output element in the requested output type.
__device__ __forceinline__ void store_out(void* out, int64_t i, int32_t dtype, float v) {
  if (dtype == PA_F32)
    static_cast<float*>(out)[i] = v;
  else if (dtype == PA_BF16)
    static_cast<__nv_bfloat16*>(out)[i] = __float2bfloat16_rn(v);
  else
    static_cast<__half*>(out)[i] = __float2half_rn(v);
}

// Store 4 consecutive output elements starting at element i (a multiple of
// 4) in the requested output type.
__device__ __forceinline__ void store_out4(void* out, int64_t i, int32_t dtype, float4 v) {
  if (dtype == PA_F32) {
    *reinterpret_cast<float4*>(static_cast<float*>(out) + i) = v;
  } else if (dtype == PA_BF16) {
    __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + i) =
        make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  } else {
    __half2 a = __floats2half2_rn(v.x, v.y), b = __floats2half2_rn(v.z, v.w);
    *reinterpret_cast<uint2*>(static_cast<uint16_t*>(out) + i) =
        make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
  }
}

// Store 16 consecutive output elements starting at element i (a multiple of
// 16; the output 16-byte aligned) in the requested output type.
__device__ __forceinline__ void store_row16(void* out, int64_t i, int32_t dtype,
                                            const float (&v)[16]) {
  if (dtype == PA_F32) {
    float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + i);
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  } else {
    uint32_t w[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      if (dtype == PA_BF16) {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __half2 h = __floats2half2_rn(v[2 * k], v[2 * k + 1]);
        w[k] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
    uint4* p = reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + i);
    p[0] = make_uint4(w[0], w[1], w[2], w[3]);
    p[1] = make_uint4(w[4], w[5], w[6], w[7]);
  }
}

// 16-bit element bits and round-to-nearest conversion, per element type.
__device__ __forceinline__ uint16_t bits16(__nv_bfloat16 x) { return __bfloat16_as_ushort(x); }
__device__ __forceinline__ uint16_t bits16(__half x) { return __half_as_ushort(x); }
__device__ __forceinline__ __nv_bfloat16 round16(float x, __nv_bfloat16*) {
  return __float2bfloat16_rn(x);
}
__device__ __forceinline__ __half round16(float x, __half*) { return __float2half_rn(x); }

// Record a device-side error in the status word (if the call has one).
__device__ __forceinline__ void set_status(int32_t* status, int32_t code) {
  if (status) atomicExch(status, code);
}

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

// Valid sequence length for this call: 0 <= L <= max_seq_len (the bound the
// caller promised, which also sizes the V2 workspace) and L <= the tokens the
// block-table row can address.
__device__ __forceinline__ bool seq_len_ok(const KernelArgs& a, int32_t L) {
  if (L < 0 || L > a.max_seq_len) return false;
  return static_cast<int64_t>(L) <= static_cast<int64_t>(a.max_blocks_per_seq) * a.block_size;
}

}  // namespace pa
