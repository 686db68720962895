// pa_prefill_host.cu -- pa_prefill: parameter checks, the five TMA tensor
// maps and the launch of the tensor-core prefill kernel (pa_prefill.cuh).
//
// Maps (all with the 128-byte swizzle):
//   q       [T, Hq, D]   as (64, Hq, T, D / 64), box (64, 1, 128, 1):
//                        one 64-element slice of 128 query rows of one head;
//   k (new) [T, Hkv, D]  the same view, box (64, 1, 128, 1);
//   v (new) [T, Hkv, D]  box (64, 1, 16, D / 64): 16 rows, slice-major;
//   k_cache              rows of D, box (64, BS): one slice of one block;
//   v_cache              (64, rows, D / 64), box (64, BS, D / 64): a whole
//                        block slice-major.
#include <cstdint>

#include "pa.h"
#include "pa_internal.h"

namespace {

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

pa_status_t check(const pa_prefill_params_t* p) {
  if (!p) return PA_ERR_INVALID_ARG;
  if (p->num_seqs < 0 || p->num_heads < 1 || p->num_kv_heads < 1) return PA_ERR_INVALID_ARG;
  if (p->num_heads % p->num_kv_heads) return PA_ERR_INVALID_ARG;
  if (p->total_tokens < 0 || p->max_query_len < 0 || p->max_ctx_len < 0) return PA_ERR_INVALID_ARG;
  if (p->block_size < 1 || p->num_blocks < 1 || p->max_blocks_per_seq < 1) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p->max_ctx_len) >
      static_cast<int64_t>(p->max_blocks_per_seq) * p->block_size)
    return PA_ERR_INVALID_ARG;
  if (!(p->scale > 0.f) || p->scale > 3.0e38f) return PA_ERR_INVALID_ARG;
  if (p->flags & ~PA_FLAG_SELFTEST_STALL) return PA_ERR_INVALID_ARG;
  if (p->kv_dtype != PA_BF16 && p->kv_dtype != PA_F16) return PA_ERR_UNSUPPORTED;
  if (p->out_dtype != PA_F32 && p->out_dtype != p->kv_dtype) return PA_ERR_INVALID_ARG;
  const int D = p->head_dim, BS = p->block_size;
  const bool shape = (D == 256 && (BS == 16 || BS == 32)) ||
                     (D == 128 && (BS == 16 || BS == 32 || BS == 64));
  if (!shape) return PA_ERR_UNSUPPORTED;
  // TMA coordinates are int32
  const int64_t rows = static_cast<int64_t>(p->num_blocks) * p->num_kv_heads * BS;
  if (rows + BS >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(p->total_tokens) + 256 >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_prefill(const pa_prefill_params_t* p, const void* q, const void* k,
                                  const void* v, const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, const int32_t* query_start,
                                  const int32_t* ctx_lens, void* out, cudaStream_t stream) {
  using namespace pa;
  pa_status_t st = check(p);
  if (st != PA_OK) return st;
  if (p->num_seqs == 0 || p->total_tokens == 0 || p->max_query_len == 0) return PA_OK;
  for (const void* ptr : {q, k, v, k_cache, v_cache, static_cast<const void*>(out)})
    if (!ptr) return PA_ERR_INVALID_ARG;
  if (!block_tables || !query_start || !ctx_lens) return PA_ERR_INVALID_ARG;
  for (const void* ptr : {q, k, v, k_cache, v_cache, static_cast<const void*>(out)})
    if (!aligned(ptr, 16)) return PA_ERR_MISALIGNED;
  if (!aligned(block_tables, 4) || !aligned(query_start, 4) || !aligned(ctx_lens, 4))
    return PA_ERR_MISALIGNED;
  const int sms = sm100_num_sms();
  if (sms <= 0) return PA_ERR_UNSUPPORTED;

  const uint64_t D = static_cast<uint64_t>(p->head_dim);
  const uint64_t T = static_cast<uint64_t>(p->total_tokens);
  const uint64_t Hq = static_cast<uint64_t>(p->num_heads), Hkv = static_cast<uint64_t>(p->num_kv_heads);
  const uint64_t BS = static_cast<uint64_t>(p->block_size);
  const uint64_t rows = static_cast<uint64_t>(p->num_blocks) * Hkv * BS;
  CUtensorMap m[5];
  {
    const uint64_t dims[4] = {64, Hq, T, D / 64};
    const uint64_t strides[3] = {D * 2, Hq * D * 2, 128};
    const uint32_t box[4] = {64, 1, 128, 1};
    if (encode_tiled(&m[0], p->kv_dtype, 4, q, dims, strides, box) != cudaSuccess)
      return PA_ERR_UNSUPPORTED;
  }
  {
    const uint64_t dims[4] = {64, Hkv, T, D / 64};
    const uint64_t strides[3] = {D * 2, Hkv * D * 2, 128};
    const uint32_t box_k[4] = {64, 1, 128, 1};
    const uint32_t box_v[4] = {64, 1, 16, static_cast<uint32_t>(D / 64)};
    if (encode_tiled(&m[1], p->kv_dtype, 4, k, dims, strides, box_k) != cudaSuccess ||
        encode_tiled(&m[2], p->kv_dtype, 4, v, dims, strides, box_v) != cudaSuccess)
      return PA_ERR_UNSUPPORTED;
  }
  {
    const uint64_t dims[2] = {D, rows};
    const uint64_t strides[1] = {D * 2};
    const uint32_t box[2] = {64, static_cast<uint32_t>(BS)};
    if (encode_tiled(&m[3], p->kv_dtype, 2, k_cache, dims, strides, box) != cudaSuccess)
      return PA_ERR_UNSUPPORTED;
  }
  {
    const uint64_t dims[3] = {64, rows, D / 64};
    const uint64_t strides[2] = {D * 2, 128};
    const uint32_t box[3] = {64, static_cast<uint32_t>(BS), static_cast<uint32_t>(D / 64)};
    if (encode_tiled(&m[4], p->kv_dtype, 3, v_cache, dims, strides, box) != cudaSuccess)
      return PA_ERR_UNSUPPORTED;
  }

  PrefillArgs a{};
  a.block_tables = block_tables;
  a.query_start = query_start;
  a.ctx_lens = ctx_lens;
  a.out = out;
  a.num_seqs = p->num_seqs;
  a.num_heads = p->num_heads;
  a.num_kv_heads = p->num_kv_heads;
  a.head_dim = p->head_dim;
  a.block_size = p->block_size;
  a.num_blocks = p->num_blocks;
  a.max_blocks_per_seq = p->max_blocks_per_seq;
  a.total_tokens = p->total_tokens;
  a.max_query_len = p->max_query_len;
  a.max_ctx_len = p->max_ctx_len;
  a.group = p->num_heads / p->num_kv_heads;
  a.out_dtype = p->out_dtype;
  a.scale_log2 = p->scale * 1.442695040888963407360f;
  a.qtiles = (p->max_query_len + 127) / 128;
  // Units cost up to ceil(max_ctx_len / 128) + qtiles key tiles.  Batches of
  // several sequences are walked by cost (longest first), as long as the
  // (level, sequence) pairs every role scans stay few.
  const int64_t levels = (static_cast<int64_t>(p->max_ctx_len) + 127) / 128 + a.qtiles;
  a.cost_levels = (p->num_seqs > 1 && levels * p->num_seqs <= 8192) ? static_cast<int32_t>(levels) : 0;
  a.selftest_stall = (p->flags & PA_FLAG_SELFTEST_STALL) ? 1 : 0;
  const cudaError_t e = p->kv_dtype == PA_BF16 ? launch_prefill_bf16(a, m, sms, stream)
                                               : launch_prefill_f16(a, m, sms, stream);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}
