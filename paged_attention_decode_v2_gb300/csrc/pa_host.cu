// pa_host.cu -- the decode step from host memory: pa_host_staging_size and
// pa_decode_host (include/pa.h).  The step's per-call inputs (q, the block
// table and the sequence lengths) are copied into caller-owned device
// staging memory, pa_decode runs on them, and `out` is copied back; the KV
// cache and the workspace stay resident on the device.  This is the one
// decode call that waits for its stream.
#include <cstdint>

#include <cuda_runtime_api.h>

#include "pa.h"
#include "pa_internal.h"

namespace pa {
namespace {

constexpr size_t kAlign = 256;

size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

size_t elem_bytes(pa_dtype_t t) { return t == PA_F32 ? 4 : 2; }

// Offsets of the staged tensors: q | block_tables | seq_lens | out, each on
// a 256-byte boundary.
struct Staging {
  size_t q_bytes, bt_bytes, sl_bytes, out_bytes;
  size_t bt_off, sl_off, out_off, total;
};

Staging staging_layout(const pa_params_t* p) {
  Staging s;
  const size_t rows = static_cast<size_t>(p->num_seqs) * static_cast<size_t>(p->num_heads);
  s.q_bytes = rows * p->head_dim * elem_bytes(p->kv_dtype);
  s.bt_bytes = static_cast<size_t>(p->num_seqs) * p->max_blocks_per_seq * sizeof(int32_t);
  s.sl_bytes = static_cast<size_t>(p->num_seqs) * sizeof(int32_t);
  s.out_bytes = rows * p->head_dim * elem_bytes(p->out_dtype);
  s.bt_off = round_up(s.q_bytes);
  s.sl_off = s.bt_off + round_up(s.bt_bytes);
  s.out_off = s.sl_off + round_up(s.sl_bytes);
  s.total = s.out_off + round_up(s.out_bytes);
  return s;
}

}  // namespace
}  // namespace pa

using namespace pa;

extern "C" {

size_t pa_host_staging_size(const pa_params_t* p) {
  if (check_params(p, false) != PA_OK) return 0;
  return staging_layout(p).total;
}

pa_status_t pa_host_staging_offsets(const pa_params_t* p, size_t offsets[5]) {
  if (!offsets || check_params(p, false) != PA_OK) return PA_ERR_INVALID_ARG;
  const Staging s = staging_layout(p);
  offsets[0] = 0;
  offsets[1] = s.bt_off;
  offsets[2] = s.sl_off;
  offsets[3] = s.out_off;
  offsets[4] = s.total;
  return PA_OK;
}

pa_status_t pa_decode_host(const pa_params_t* p, const void* q_host, const void* k_cache,
                           const void* v_cache, const int32_t* block_tables_host,
                           const int32_t* seq_lens_host, void* workspace, size_t workspace_bytes,
                           void* staging, size_t staging_bytes, void* out_host,
                           cudaStream_t stream) {
  pa_status_t st = check_params(p, false);
  if (st != PA_OK) return st;
  if (!staging || !out_host) return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(staging) % kAlign) return PA_ERR_MISALIGNED;
  const Staging s = staging_layout(p);
  if (staging_bytes < s.total) return PA_ERR_WORKSPACE_TOO_SMALL;
  if (p->num_seqs > 0 && (!q_host || !block_tables_host || !seq_lens_host))
    return PA_ERR_INVALID_ARG;
  // everything pa_decode checks, before anything is enqueued
  if (pa_decode_path(p) == 2) {
    if (!workspace) return PA_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % kAlign) return PA_ERR_MISALIGNED;
    if (workspace_bytes < pa_workspace_size(p)) return PA_ERR_WORKSPACE_TOO_SMALL;
  } else if (pa_decode_path(p) != 1) {
    return PA_ERR_INVALID_ARG;
  }
  if (!k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(k_cache) % 16 || reinterpret_cast<uintptr_t>(v_cache) % 16)
    return PA_ERR_MISALIGNED;

  uint8_t* base = static_cast<uint8_t*>(staging);
  void* q_d = base;
  int32_t* bt_d = reinterpret_cast<int32_t*>(base + s.bt_off);
  int32_t* sl_d = reinterpret_cast<int32_t*>(base + s.sl_off);
  void* out_d = base + s.out_off;
  // From here on copies may be queued that read the caller's host buffers:
  // an error return first waits for the stream, so that no copy still reads
  // (or writes) them after the call has returned.
  auto fail = [&](pa_status_t e) {
    cudaStreamSynchronize(stream);
    return e;
  };
  if (p->num_seqs > 0) {
    const char* qh = static_cast<const char*>(q_host);
    const bool mirrored = reinterpret_cast<const char*>(block_tables_host) == qh + s.bt_off &&
                          reinterpret_cast<const char*>(seq_lens_host) == qh + s.sl_off;
    if (mirrored) {  // the host inputs already have the staging layout: one copy
      if (cudaMemcpyAsync(q_d, q_host, s.sl_off + s.sl_bytes, cudaMemcpyHostToDevice, stream) !=
          cudaSuccess)
        return fail(PA_ERR_CUDA);
    } else if (cudaMemcpyAsync(q_d, q_host, s.q_bytes, cudaMemcpyHostToDevice, stream) !=
                   cudaSuccess ||
               cudaMemcpyAsync(bt_d, block_tables_host, s.bt_bytes, cudaMemcpyHostToDevice,
                               stream) != cudaSuccess ||
               cudaMemcpyAsync(sl_d, seq_lens_host, s.sl_bytes, cudaMemcpyHostToDevice, stream) !=
                   cudaSuccess) {
      return fail(PA_ERR_CUDA);
    }
  }
  st = pa_decode(p, q_d, k_cache, v_cache, bt_d, sl_d, workspace, workspace_bytes, out_d, stream);
  if (st != PA_OK) return fail(st);
  if (p->num_seqs > 0 &&
      cudaMemcpyAsync(out_host, out_d, s.out_bytes, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
    return fail(PA_ERR_CUDA);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return PA_ERR_CUDA;
  return PA_OK;
}

}  // extern "C"
