// pa_tc_host.cu -- host side of the tensor-core path: when it applies, and
// the TMA tensor maps of the two caches.
//
// The caches are viewed as rows of head_dim elements, one row per
// (block, KV head, slot): row = (block * num_kv_heads + kv_head) *
// block_size + slot.  Keys use a 2-D map (head_dim, rows) with a 64 x
// block_size box, so one copy brings one 64-element slice of one block;
// values use a 3-D map (64, rows, head_dim / 64) whose box is a whole block
// laid out slice-major; q is viewed as (head_dim, num_seqs * num_heads)
// rows with an 8-row box (one KV head's query rows).  All use the 128-byte
// swizzle the MMA descriptors expect.
#include <cstring>
#include <atomic>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "pa_internal.h"

namespace pa {

cudaError_t launch_tc_bf16(const KernelArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           const CUtensorMap& qmap, const CUtensorMap& pmap, bool v2, int num_sms,
                           cudaStream_t s);
cudaError_t launch_tc_f16(const KernelArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                          const CUtensorMap& qmap, const CUtensorMap& pmap, bool v2, int num_sms,
                          cudaStream_t s);
cudaError_t launch_sx_bf16(const KernelArgs& a, const CUtensorMap& pmap, bool v2, cudaStream_t s);
cudaError_t launch_sx_f16(const KernelArgs& a, const CUtensorMap& pmap, bool v2, cudaStream_t s);

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static std::once_flag once;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct DeviceInfo {
  int state = 0;  // 0 unknown, 1 runs the sm_100-family kernels, 2 does not
  int num_sms = 0;
};

// Per-device attributes, queried on first use.  Callers on several host
// threads may race to fill an entry; they store the same values, and the
// entry is published by its atomic state after the SM count.
DeviceInfo device_info() {
  static std::atomic<int> state[128];
  static std::atomic<int> num_sms[128];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 128) return DeviceInfo{};
  int st = state[dev].load(std::memory_order_acquire);
  if (!st) {
    int major = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    num_sms[dev].store(sms, std::memory_order_relaxed);
    st = (major == 10 && sms > 0) ? 1 : 2;
    state[dev].store(st, std::memory_order_release);
  }
  return DeviceInfo{st, num_sms[dev].load(std::memory_order_relaxed)};
}

}  // namespace

cudaError_t encode_tiled(CUtensorMap* map, pa_dtype_t dtype, uint32_t rank, const void* base,
                         const uint64_t* dims, const uint64_t* strides, const uint32_t* box) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const CUtensorMapDataType dt =
      dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (uint32_t i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return enc(map, dt, rank, const_cast<void*>(base), d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? cudaSuccess
             : cudaErrorInvalidValue;
}

int sm100_num_sms() {
  const DeviceInfo d = device_info();
  return d.state == 1 ? d.num_sms : 0;
}

bool tc_applicable(const pa_params_t* p) {
  if (p->flags & (PA_FLAG_PORTABLE | PA_FLAG_SPLIT_X)) return false;
  if (p->kv_dtype != PA_BF16 && p->kv_dtype != PA_F16) return false;
  if (p->num_heads / p->num_kv_heads > 8) return false;
  const int D = p->head_dim, BS = p->block_size;
  const bool shape = (D == 256 && (BS == 16 || BS == 32)) ||
                     (D == 128 && (BS == 16 || BS == 32 || BS == 64));
  if (!shape) return false;
  const int64_t rows = static_cast<int64_t>(p->num_blocks) * p->num_kv_heads * BS;
  if (rows + BS >= (int64_t(1) << 31)) return false;  // TMA row coordinates are int32
  if (static_cast<int64_t>(p->num_seqs) * p->num_heads + 8 >= (int64_t(1) << 31)) return false;
  return encoder() != nullptr && device_info().state == 1;
}

bool sx_applicable(const pa_params_t* p) {
  if ((p->flags & PA_FLAG_SPLIT_X) == 0 || (p->flags & PA_FLAG_PORTABLE)) return false;
  if (p->kv_dtype != PA_BF16 && p->kv_dtype != PA_F16) return false;
  if (p->num_heads / p->num_kv_heads > 8) return false;
  const int D = p->head_dim, BS = p->block_size;
  if (!(D == 64 || D == 128 || D == 256) || !(BS == 16 || BS == 32)) return false;
  return device_info().state == 1;
}

// The V2 partials as [rows][NP][head_dim] floats, a box of 32 elements x up
// to 256 partitions of one row: the tile copies of the one-launch grid's
// reduce units.
static bool encode_partials_map(PFN_cuTensorMapEncodeTiled_v12000 enc, const KernelArgs& a,
                                CUtensorMap* pmap) {
  const cuuint64_t D = static_cast<cuuint64_t>(a.head_dim);
  const cuuint64_t np = static_cast<cuuint64_t>(a.num_partitions);
  const cuuint64_t dims[3] = {D, np, static_cast<cuuint64_t>(a.num_seqs) * a.num_heads};
  const cuuint64_t strides[2] = {D * 4, np * D * 4};
  const cuuint32_t box[3] = {32, static_cast<cuuint32_t>(np < 256 ? np : 256), 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(pmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, a.tmp_out, dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The split-x kernel reads the caches by bulk copy (one contiguous run per
// block and KV head); only the one-launch grid needs a tensor map (the
// partials).
cudaError_t launch_sx(const KernelArgs& a, pa_dtype_t kv, bool v2, cudaStream_t s) {
  CUtensorMap pmap;
  std::memset(&pmap, 0, sizeof pmap);  // never read unless a.fused
  if (a.fused) {
    auto enc = encoder();
    if (!enc) return cudaErrorNotSupported;
    if (!encode_partials_map(enc, a, &pmap)) return cudaErrorInvalidValue;
  }
  return kv == PA_BF16 ? launch_sx_bf16(a, pmap, v2, s) : launch_sx_f16(a, pmap, v2, s);
}

cudaError_t launch_tc(const KernelArgs& a, pa_dtype_t kv, bool v2, cudaStream_t s) {
  auto enc = encoder();
  if (!enc) return cudaErrorNotSupported;
  const CUtensorMapDataType dt =
      kv == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint64_t D = static_cast<cuuint64_t>(a.head_dim);
  const cuuint64_t rows = static_cast<cuuint64_t>(a.num_blocks) * a.num_kv_heads * a.block_size;
  const cuuint32_t BS = static_cast<cuuint32_t>(a.block_size);
  CUtensorMap kmap, vmap;
  {
    const cuuint64_t dims[2] = {D, rows};
    const cuuint64_t strides[1] = {D * 2};
    const cuuint32_t box[2] = {64, BS};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&kmap, dt, 2, const_cast<void*>(a.k_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {
    const cuuint64_t dims[3] = {64, rows, D / 64};
    const cuuint64_t strides[2] = {D * 2, 128};
    const cuuint32_t box[3] = {64, BS, static_cast<cuuint32_t>(D / 64)};
    const cuuint32_t es[3] = {1, 1, 1};
    if (enc(&vmap, dt, 3, const_cast<void*>(a.v_cache), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  CUtensorMap qmap;
  {
    const cuuint64_t dims[2] = {D, static_cast<cuuint64_t>(a.num_seqs) * a.num_heads};
    const cuuint64_t strides[1] = {D * 2};
    const cuuint32_t box[2] = {64, 8};
    const cuuint32_t es[2] = {1, 1};
    if (enc(&qmap, dt, 2, const_cast<void*>(a.q), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  // only the one-launch V2 grid reads the partials map; otherwise a copy of
  // the q map stands in, never used
  CUtensorMap pmap = qmap;
  if (a.fused && !encode_partials_map(enc, a, &pmap)) return cudaErrorInvalidValue;
  const int sms = device_info().num_sms;
  return kv == PA_BF16 ? launch_tc_bf16(a, kmap, vmap, qmap, pmap, v2, sms, s)
                       : launch_tc_f16(a, kmap, vmap, qmap, pmap, v2, sms, s);
}

}  // namespace pa
