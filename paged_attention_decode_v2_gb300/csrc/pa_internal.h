// pa_internal.h -- internal interface between the C ABI (pa_api.cu) and the
// kernels.  Not installed; users include include/pa.h only.
#pragma once

#include <cstdint>

#include <cuda.h>
#include <cuda_runtime_api.h>

#include "pa.h"

namespace pa {

// Everything a kernel needs, passed by value as one kernel parameter.
struct KernelArgs {
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  void* out;            // final output (V1 kernels, V2 reduce)
  float* max_logits;    // V2 workspace regions
  float* exp_sums;
  float* tmp_out;
  int32_t* status;      // V2 status word, or nullptr (V1)
  int32_t num_seqs;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t max_seq_len;
  int32_t partition_size;  // V2: tokens per partition
  int32_t num_partitions;  // V2: NP = ceil(max_seq_len / partition_size)
  int32_t group;           // G = num_heads / num_kv_heads
  int32_t out_dtype;       // pa_dtype_t
  float scale_log2;        // scale * log2(e): logits are kept in base-2 units
  int32_t selftest_stall;  // PA_FLAG_SELFTEST_STALL was given
  int32_t split_x;         // PA_FLAG_SPLIT_X: the pages' V1 cache layout
  int32_t single_direct;   // V2 pass 1 + reduce in one call: a sequence of at most
                           // partition_size tokens is finished by pass 1 (written
                           // straight into out) and the reduce skips its rows
};

// Everything the prefill kernel needs besides its tensor maps (pa_prefill.cuh).
struct PrefillArgs {
  const int32_t* block_tables;
  const int32_t* query_start;
  const int32_t* ctx_lens;
  void* out;
  int32_t num_seqs;
  int32_t num_heads;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t block_size;
  int32_t num_blocks;
  int32_t max_blocks_per_seq;
  int32_t total_tokens;
  int32_t max_query_len;
  int32_t max_ctx_len;
  int32_t group;        // G = num_heads / num_kv_heads
  int32_t out_dtype;    // pa_dtype_t
  float scale_log2;     // scale * log2(e)
  int32_t qtiles;       // ceil(max_query_len / 128)
  int32_t cost_levels;  // > 0: walk units by cost, from this level down (0: by query tile)
  int32_t selftest_stall;
};

// Launchers return cudaSuccess or the launch error.
cudaError_t launch_generic_f32(const KernelArgs& a, bool v2, cudaStream_t s);
cudaError_t launch_generic_bf16(const KernelArgs& a, bool v2, cudaStream_t s);
cudaError_t launch_generic_f16(const KernelArgs& a, bool v2, cudaStream_t s);
cudaError_t launch_reduce(const KernelArgs& a, cudaStream_t s, bool pdl);
// Parameter checks of every decode entry point (`v2`: the partition rules too).
pa_status_t check_params(const pa_params_t* p, bool v2);

// Tensor-core path (pa_tc_host.cu): whether it serves these parameters on
// the current device, and its launch (pass 1 for V2, the whole pass for V1).
bool tc_applicable(const pa_params_t* p);
cudaError_t launch_tc(const KernelArgs& a, pa_dtype_t kv, bool v2, cudaStream_t s);

// TMA tiled tensor map (pa_tc_host.cu) with the 128-byte swizzle the MMA
// descriptors expect: `rank` dims (innermost first), the byte strides of
// dims 1..rank-1 and the box.  cudaErrorNotSupported without the driver
// entry point, cudaErrorInvalidValue if the driver rejects the map.
cudaError_t encode_tiled(CUtensorMap* map, pa_dtype_t dtype, uint32_t rank, const void* base,
                         const uint64_t* dims, const uint64_t* strides, const uint32_t* box);
// SMs of the current device if it runs the sm_100-family kernels, else 0.
int sm100_num_sms();

// Prefill launches (pa_prefill_bf16.cu / pa_prefill_f16.cu); maps: q, chunk
// keys, chunk values, key cache, value cache.
cudaError_t launch_prefill_bf16(const PrefillArgs& a, const CUtensorMap (&m)[5], int num_sms,
                                cudaStream_t s);
cudaError_t launch_prefill_f16(const PrefillArgs& a, const CUtensorMap (&m)[5], int num_sms,
                               cudaStream_t s);

// Workspace carve-up shared by pa_workspace_size and the V2 launch.
struct WorkspaceLayout {
  size_t max_logits_off, exp_sums_off, tmp_out_off, total;
};
WorkspaceLayout workspace_layout(int64_t num_seqs, int64_t num_heads, int64_t head_dim,
                                 int64_t num_partitions);

}  // namespace pa
