// pa_static.cu -- pa_decode_v2_static: the V2 decode with its workspace in a
// fixed-size device array that the library holds, for callers that cannot
// allocate device memory themselves.
//
// Some callers have no way to call cudaMalloc (or any allocator) at the
// point where they decode: a plugin inside a host runtime that owns every
// device allocation and forbids raw ones, a C program that links libpa
// without torch or any other allocator, or a real-time loop that must not
// risk an allocation failure or an allocator stall mid-run.  This entry
// point lets them run V2 with nothing but their inputs and outputs.
//
// The array below lives in the library's device image: every GPU on which
// libpa.so's code is loaded holds PA_STATIC_WORKSPACE_BYTES of device memory
// for it until the process exits.  All calls on a device share it and it
// keeps whatever the last call left there.  V2 only reads back the partials
// the same call wrote; the one part that must be initialised is the control
// block (the counters of the one-launch step), which the first call in a
// context initialises on its stream and every launch leaves ready for the
// next.  Two calls that overlap on the
// GPU (different streams, or different host threads, without ordering
// between them) race on it: order them on one stream.
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime_api.h>

#include "pa.h"
#include "pa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_ws[PA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 128;

// The driver calls that name the current context, looked up once through the
// runtime (the library links no driver library of its own).
struct CtxCalls {
  PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
  PFN_cuCtxGetId_v12000 get_id = nullptr;
};

const CtxCalls& ctx_calls() {
  static std::once_flag once;
  static CtxCalls c;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      c.get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      c.get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
  });
  return c;
}

// Unique id of the calling thread's current context (0 if there is none
// yet, or the driver cannot tell).
unsigned long long current_ctx_id() {
  const CtxCalls& c = ctx_calls();
  if (!c.get_current || !c.get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (c.get_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
  if (c.get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

std::mutex g_mu;
struct Cached {
  unsigned long long ctx = 0;  // context the address belongs to (0: none cached)
  void* addr = nullptr;
};
Cached g_ws[kMaxDevices];

// Host code cannot use g_static_ws's address directly (on the host it names
// a stand-in, not device memory), so it is looked up with the device
// current and cached.  The module, and so the address, belongs to one
// context: the cache is keyed on the current context's unique id, and a new
// context on the device (after cudaDeviceReset, or a driver-API context
// made current by the caller) gets its own lookup.  With each lookup the
// control block (status word, marker and counters) is initialised on
// `stream`, as pa_workspace_init does for a caller's workspace.
pa_status_t static_ws_address(void** out, cudaStream_t stream) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  unsigned long long ctx = current_ctx_id();
  if (ctx != 0 && g_ws[dev].ctx == ctx) {
    *out = g_ws[dev].addr;
    return PA_OK;
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_static_ws) != cudaSuccess || !p) return PA_ERR_CUDA;
  if (pa_workspace_init(p, pa::kCtrlBytes, stream) != PA_OK) return PA_ERR_CUDA;
  // the lookup makes the device's primary context current if nothing was
  if (ctx == 0) ctx = current_ctx_id();
  g_ws[dev].ctx = ctx;  // 0 when the id is unknown: looked up again next call
  g_ws[dev].addr = p;
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_decode_v2_static(const pa_params_t* params, const void* q,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, const int32_t* seq_lens,
                                           void* out, cudaStream_t stream) {
  const size_t need = pa_workspace_size(params);
  if (need == 0)  // invalid parameters: let the regular checks name the problem
    return pa_decode_v2(params, q, k_cache, v_cache, block_tables, seq_lens, nullptr, 0, out,
                        stream);
  if (need > PA_STATIC_WORKSPACE_BYTES) return PA_ERR_WORKSPACE_TOO_SMALL;
  if (params->num_seqs == 0) return PA_OK;
  void* ws = nullptr;
  const pa_status_t st = static_ws_address(&ws, stream);
  if (st != PA_OK) return st;
  return pa_decode_v2(params, q, k_cache, v_cache, block_tables, seq_lens, ws,
                      PA_STATIC_WORKSPACE_BYTES, out, stream);
}
