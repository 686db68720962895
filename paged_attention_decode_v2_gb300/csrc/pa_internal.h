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
  int32_t fused;           // V2 in one launch: the pass-1 grid runs pass 2 itself
                           // after its streaming (pa_grid_reduce.cuh)
};

// The workspace starts with a control block of fixed size: the status word,
// an initialisation marker, and the words of the one-launch V2 step (start
// counter, finished counters, reduce-unit queue).  It sits at the same place
// with the same size whatever the parameters; pa_workspace_init zeroes it and
// writes the marker, and a one-launch V2 step run on a workspace without the
// marker merges nothing: it reports PA_ERR_WORKSPACE_NOT_INIT and the rows it
// would have reduced become NaN.
constexpr size_t kCtrlBytes = PA_WORKSPACE_CONTROL_BYTES;
constexpr size_t kMarkerOffset = 4;
constexpr size_t kSyncOffset = 256;
constexpr int kMarkerByte = 0x5A;
constexpr int32_t kMarker = 0x5A5A5A5A;

// Persistent grid of the tensor-core pass-1 kernel for `items` work items
// (0 when there are fewer items than SMs: the one-CTA-per-SM shape runs
// instead).  At most two CTAs per SM; with a dense item walk (`compact`
// false) the grid is sized so every CTA does the same number of rounds.
inline int64_t tc_persistent_grid(int64_t items, bool compact, int num_sms) {
  if (items < num_sms) return 0;
  const int64_t slots = static_cast<int64_t>(num_sms) * 2;
  int64_t grid = items < slots ? items : slots;
  if (!compact && items > slots) {
    const int64_t rounds = (items + slots - 1) / slots;
    grid = (items + rounds - 1) / rounds;
  }
  return grid;
}

// Whether the V2 step runs as one launch: the persistent tensor-core grid
// takes at most one reduce unit (query row x 32 elements of head_dim) per
// CTA, so its own CTAs run pass 2 in one round after their streaming; other
// batches use the dependent reduce kernel, which has more CTAs in flight.
// Both tensor-core kernels (either cache layout) size their grids this way.
inline bool one_launch_plan(int64_t num_seqs, int64_t num_heads, int64_t num_kv_heads,
                            int64_t head_dim, int64_t np, int num_sms) {
  const int64_t items = num_seqs * num_kv_heads * np;
  const bool compact = num_seqs > 1 && num_seqs <= 1024;  // the kernels' compact work list
  const int64_t grid = tc_persistent_grid(items, compact, num_sms);
  // a unit holds the statistics of up to 1024 partitions
  return grid > 0 && np <= 1024 && num_seqs * num_heads * (head_dim / 32) <= grid;
}

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
// Tensor-core path for caches in the split-x layout (pa_sx.cuh, launched
// from pa_tc_host.cu): whether it serves these parameters on the current
// device, and its launch (pass 1 for V2, or the whole V2 step when
// a.fused; the whole pass for V1).
bool sx_applicable(const pa_params_t* p);
cudaError_t launch_sx(const KernelArgs& a, pa_dtype_t kv, bool v2, cudaStream_t s);

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
