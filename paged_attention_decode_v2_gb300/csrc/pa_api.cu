// pa_api.cu -- the C ABI declared in include/pa.h: argument checks, the V1 /
// V2 dispatch, workspace carve-up and kernel launches.  No allocation, no
// synchronisation (except pa_read_device_status, which says so).
#include <cstdint>
#include <cstring>

#include <cuda_runtime_api.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa {

namespace {

constexpr int32_t kDefaultV1MaxSeqLen = 8192;  // threshold on the pages
constexpr size_t kAlign = 256;
constexpr float kLog2eHost = 1.442695040888963407360f;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool aligned(const void* p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) % n) == 0; }

}  // namespace

// Checks shared by every decode entry point; `v2` adds the partition rules.
pa_status_t check_params(const pa_params_t* p, bool v2) {
  if (!p) return PA_ERR_INVALID_ARG;
  if (p->num_seqs < 0 || p->num_heads < 1 || p->num_kv_heads < 1) return PA_ERR_INVALID_ARG;
  if (p->num_heads % p->num_kv_heads) return PA_ERR_INVALID_ARG;
  if (p->head_dim < 1 || p->block_size < 1 || p->num_blocks < 1) return PA_ERR_INVALID_ARG;
  if (p->max_blocks_per_seq < 1 || p->max_seq_len < 0) return PA_ERR_INVALID_ARG;
  if (static_cast<int64_t>(p->max_seq_len) >
      static_cast<int64_t>(p->max_blocks_per_seq) * p->block_size)
    return PA_ERR_INVALID_ARG;
  if (p->flags & ~(PA_FLAG_PORTABLE | PA_FLAG_SELFTEST_STALL | PA_FLAG_SPLIT_X))
    return PA_ERR_INVALID_ARG;
  if (p->kv_dtype != PA_F32 && p->kv_dtype != PA_BF16 && p->kv_dtype != PA_F16)
    return PA_ERR_UNSUPPORTED;
  if (p->out_dtype != PA_F32 && p->out_dtype != p->kv_dtype) return PA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256) return PA_ERR_UNSUPPORTED;
  if (p->num_heads > 65535 || p->num_kv_heads > 65535 || p->num_seqs > 65535)
    return PA_ERR_UNSUPPORTED;
  if (v2) {
    if (p->partition_size < 1 || p->partition_size % p->block_size) return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

namespace {

int32_t threshold(const pa_params_t* p) {
  return p->v1_max_seq_len > 0 ? p->v1_max_seq_len : kDefaultV1MaxSeqLen;
}

int64_t num_partitions(const pa_params_t* p) {
  const int64_t n = (static_cast<int64_t>(p->max_seq_len) + p->partition_size - 1) /
                    p->partition_size;
  return n > 0 ? n : 1;
}

pa_status_t check_tensors(const void* q, const void* k, const void* v, const int32_t* bt,
                          const int32_t* sl, const void* out) {
  if (!q || !k || !v || !bt || !sl || !out) return PA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16))
    return PA_ERR_MISALIGNED;
  if (!aligned(bt, 4) || !aligned(sl, 4)) return PA_ERR_MISALIGNED;
  return PA_OK;
}

KernelArgs make_args(const pa_params_t* p, const void* q, const void* k, const void* v,
                     const int32_t* bt, const int32_t* sl, void* out) {
  KernelArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k_cache = k;
  a.v_cache = v;
  a.block_tables = bt;
  a.seq_lens = sl;
  a.out = out;
  a.num_seqs = p->num_seqs;
  a.num_heads = p->num_heads;
  a.num_kv_heads = p->num_kv_heads;
  a.head_dim = p->head_dim;
  a.block_size = p->block_size;
  a.num_blocks = p->num_blocks;
  a.max_blocks_per_seq = p->max_blocks_per_seq;
  a.max_seq_len = p->max_seq_len;
  a.partition_size = p->partition_size;
  a.group = p->num_heads / p->num_kv_heads;
  a.out_dtype = p->out_dtype;
  a.scale_log2 = p->scale * kLog2eHost;
  a.selftest_stall = (p->flags & PA_FLAG_SELFTEST_STALL) ? 1 : 0;
  a.split_x = (p->flags & PA_FLAG_SPLIT_X) ? 1 : 0;
  return a;
}

cudaError_t launch_pass(const pa_params_t* p, const KernelArgs& a, bool v2, cudaStream_t s) {
  if (tc_applicable(p)) return launch_tc(a, p->kv_dtype, v2, s);
  if (sx_applicable(p))
    return launch_sx(a, p->kv_dtype, v2, s);
  switch (p->kv_dtype) {
    case PA_F32: return launch_generic_f32(a, v2, s);
    case PA_BF16: return launch_generic_bf16(a, v2, s);
    default: return launch_generic_f16(a, v2, s);
  }
}

}  // namespace

WorkspaceLayout workspace_layout(int64_t num_seqs, int64_t num_heads, int64_t head_dim,
                                 int64_t np) {
  WorkspaceLayout w;
  const size_t rows = static_cast<size_t>(num_seqs) * static_cast<size_t>(num_heads);
  w.max_logits_off = kCtrlBytes;  // the control block comes first
  w.exp_sums_off = w.max_logits_off + round_up(rows * np * sizeof(float));
  w.tmp_out_off = w.exp_sums_off + round_up(rows * np * sizeof(float));
  w.total = w.tmp_out_off + round_up(rows * np * head_dim * sizeof(float));
  return w;
}

}  // namespace pa

using namespace pa;

extern "C" {

size_t pa_workspace_size(const pa_params_t* p) {
  if (check_params(p, true) != PA_OK) return 0;
  return workspace_layout(p->num_seqs, p->num_heads, p->head_dim, num_partitions(p)).total;
}

int pa_decode_path(const pa_params_t* p) {
  if (check_params(p, false) != PA_OK) return 0;
  if (p->max_seq_len > threshold(p)) return check_params(p, true) == PA_OK ? 2 : 0;
  return 1;
}

pa_status_t pa_decode_v1(const pa_params_t* p, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* seq_lens, void* out, cudaStream_t stream) {
  pa_status_t st = check_params(p, false);
  if (st != PA_OK) return st;
  if (p->num_seqs == 0) return PA_OK;
  st = check_tensors(q, k_cache, v_cache, block_tables, seq_lens, out);
  if (st != PA_OK) return st;
  KernelArgs a = make_args(p, q, k_cache, v_cache, block_tables, seq_lens, out);
  if (launch_pass(p, a, false, stream) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"

namespace {

// Checks and workspace carve-up shared by the V2 entry points.  `need_in`
// is false for the reduce-only call (no q / caches / block table).
pa_status_t prepare_v2(const pa_params_t* p, const void* q, const void* k, const void* v,
                       const int32_t* bt, const int32_t* sl, const void* workspace,
                       size_t workspace_bytes, void* out, bool need_in, bool need_out,
                       KernelArgs* a) {
  pa_status_t st = check_params(p, true);
  if (st != PA_OK) return st;
  if (p->num_seqs == 0) return PA_OK;
  if (need_in) {
    st = check_tensors(q, k, v, bt, sl, need_out ? out : q);
    if (st != PA_OK) return st;
  } else {
    if (!sl || !out) return PA_ERR_INVALID_ARG;
    if (!aligned(sl, 4) || !aligned(out, 16)) return PA_ERR_MISALIGNED;
  }
  if (!workspace) return PA_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return PA_ERR_MISALIGNED;
  const int64_t np = num_partitions(p);
  if (np > 0x7fffffffLL) return PA_ERR_UNSUPPORTED;
  const WorkspaceLayout w = workspace_layout(p->num_seqs, p->num_heads, p->head_dim, np);
  if (workspace_bytes < w.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  *a = make_args(p, q, k, v, bt, sl, out);
  char* base = static_cast<char*>(const_cast<void*>(workspace));
  a->status = reinterpret_cast<int32_t*>(base);
  a->max_logits = reinterpret_cast<float*>(base + w.max_logits_off);
  a->exp_sums = reinterpret_cast<float*>(base + w.exp_sums_off);
  a->tmp_out = reinterpret_cast<float*>(base + w.tmp_out_off);
  a->num_partitions = static_cast<int32_t>(np);
  return PA_OK;
}

// Whether the V2 step runs as one launch (the pass-1 grid running pass 2
// itself): the tensor-core kernel serves these parameters as a persistent
// grid with at least one CTA per reduce unit (pa_internal.h).
bool one_launch_v2(const pa_params_t* p, int64_t np) {
  if (!tc_applicable(p) && !sx_applicable(p)) return false;
  return one_launch_plan(p->num_seqs, p->num_heads, p->num_kv_heads, p->head_dim, np,
                         sm100_num_sms());
}

}  // namespace

extern "C" {

pa_status_t pa_decode_v2(const pa_params_t* p, const void* q, const void* k_cache,
                         const void* v_cache, const int32_t* block_tables,
                         const int32_t* seq_lens, void* workspace, size_t workspace_bytes,
                         void* out, cudaStream_t stream) {
  KernelArgs a;
  pa_status_t st = prepare_v2(p, q, k_cache, v_cache, block_tables, seq_lens, workspace,
                              workspace_bytes, out, true, true, &a);
  if (st != PA_OK || p->num_seqs == 0) return st;
  // per-sequence choice inside the one pass-1 launch: sequences that fit one
  // partition are finished there, the rest are split and reduced
  a.single_direct = 1;
  if (one_launch_v2(p, a.num_partitions)) {
    // pass 2 runs in the pass-1 grid: one launch
    a.fused = 1;
    return launch_pass(p, a, true, stream) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
  }
  if (launch_pass(p, a, true, stream) != cudaSuccess) return PA_ERR_CUDA;
  if (launch_reduce(a, stream, true) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_decode_v2_partitions(const pa_params_t* p, const void* q, const void* k_cache,
                                    const void* v_cache, const int32_t* block_tables,
                                    const int32_t* seq_lens, void* workspace,
                                    size_t workspace_bytes, cudaStream_t stream) {
  KernelArgs a;
  pa_status_t st = prepare_v2(p, q, k_cache, v_cache, block_tables, seq_lens, workspace,
                              workspace_bytes, nullptr, true, false, &a);
  if (st != PA_OK || p->num_seqs == 0) return st;
  if (launch_pass(p, a, true, stream) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_decode_v2_reduce(const pa_params_t* p, const int32_t* seq_lens,
                                const void* workspace, size_t workspace_bytes, void* out,
                                cudaStream_t stream) {
  KernelArgs a;
  pa_status_t st = prepare_v2(p, nullptr, nullptr, nullptr, nullptr, seq_lens, workspace,
                              workspace_bytes, out, false, true, &a);
  if (st != PA_OK || p->num_seqs == 0) return st;
  if (launch_reduce(a, stream, false) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_decode(const pa_params_t* p, const void* q, const void* k_cache,
                      const void* v_cache, const int32_t* block_tables, const int32_t* seq_lens,
                      void* workspace, size_t workspace_bytes, void* out, cudaStream_t stream) {
  pa_status_t st = check_params(p, false);
  if (st != PA_OK) return st;
  if (p->max_seq_len > threshold(p))
    return pa_decode_v2(p, q, k_cache, v_cache, block_tables, seq_lens, workspace,
                        workspace_bytes, out, stream);
  return pa_decode_v1(p, q, k_cache, v_cache, block_tables, seq_lens, out, stream);
}

int pa_decode_launches(const pa_params_t* p) {
  if (check_params(p, false) != PA_OK) return 0;
  if (p->num_seqs == 0) return 0;
  if (p->max_seq_len <= threshold(p)) return 1;
  if (check_params(p, true) != PA_OK) return 0;
  return one_launch_v2(p, num_partitions(p)) ? 1 : 2;
}

int pa_decode_kernel(const pa_params_t* p) {
  if (check_params(p, false) != PA_OK) return 0;
  return tc_applicable(p) || sx_applicable(p) ? 2 : 1;
}

const char* pa_status_string(pa_status_t s) {
  switch (s) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported configuration";
    case PA_ERR_MISALIGNED: return "misaligned pointer";
    case PA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_DEVICE_TIMEOUT: return "device wait timed out";
    case PA_ERR_BAD_BLOCK_ID: return "block id outside the pool";
    case PA_ERR_BAD_SEQ_LEN: return "sequence length outside 0..max_seq_len";
    case PA_ERR_WORKSPACE_NOT_INIT: return "workspace not initialised (pa_workspace_init)";
  }
  return "unknown status";
}

pa_status_t pa_workspace_init(void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (!workspace || workspace_bytes < sizeof(int32_t)) return PA_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return PA_ERR_MISALIGNED;
  const size_t n = workspace_bytes < kCtrlBytes ? workspace_bytes : kCtrlBytes;
  if (cudaMemsetAsync(workspace, 0, n, stream) != cudaSuccess) return PA_ERR_CUDA;
  if (n >= kMarkerOffset + 4 &&
      cudaMemsetAsync(static_cast<char*>(workspace) + kMarkerOffset, kMarkerByte, 4, stream) !=
          cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

pa_status_t pa_read_device_status(const void* workspace, int32_t* status, int clear,
                                  cudaStream_t stream) {
  if (!workspace || !status) return PA_ERR_INVALID_ARG;
  if (!aligned(workspace, kAlign)) return PA_ERR_MISALIGNED;
  int32_t host = 0;
  if (cudaMemcpyAsync(&host, workspace, sizeof host, cudaMemcpyDeviceToHost, stream) !=
      cudaSuccess)
    return PA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
  *status = host;
  if (clear &&
      cudaMemsetAsync(const_cast<void*>(workspace), 0, sizeof(int32_t), stream) != cudaSuccess)
    return PA_ERR_CUDA;
  return PA_OK;
}

int pa_version(void) { return 100; }

}  // extern "C"
