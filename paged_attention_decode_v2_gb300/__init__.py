"""Python binding of libpa: paged single-token decode attention on GB300.

Argument marshalling only.  Every step of the computation runs in the CUDA
kernels of ``libpa.so`` behind the C ABI of ``include/pa.h``; this module
turns torch tensors into pointers and sizes, passes the current CUDA stream,
and raises :class:`PaError` on a non-OK status.  There is no fallback: if
``libpa.so`` has not been built, every call raises.

Functions mirror the C entry points: :func:`workspace_size`,
:func:`decode_v1`, :func:`decode_v2`, :func:`decode`, :func:`decode_host`,
:func:`decode_path`, :func:`status_string`, :func:`workspace_init`,
:func:`read_device_status`.
"""
from __future__ import annotations

import ctypes
import os
import threading

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpa.so")

PA_OK = 0
PA_ERR_INVALID_ARG = 1
PA_ERR_UNSUPPORTED = 2
PA_ERR_MISALIGNED = 3
PA_ERR_WORKSPACE_TOO_SMALL = 4
PA_ERR_CUDA = 5
PA_ERR_DEVICE_TIMEOUT = 6
PA_ERR_BAD_BLOCK_ID = 7
PA_ERR_BAD_SEQ_LEN = 8
PA_ERR_WORKSPACE_NOT_INIT = 9

PA_F32, PA_BF16, PA_F16 = 0, 1, 2
PA_FLAG_PORTABLE = 1
PA_FLAG_SELFTEST_STALL = 2
PA_FLAG_SPLIT_X = 4
DEFAULT_V1_MAX_SEQ_LEN = 8192

# Every symbol include/pa.h declares.
EXPORTS = ("pa_workspace_size", "pa_decode_v1", "pa_decode_v2", "pa_decode_v2_partitions",
           "pa_decode_v2_reduce", "pa_decode", "pa_decode_path", "pa_status_string",
           "pa_workspace_init", "pa_read_device_status", "pa_version", "pa_decode_v2_static",
           "pa_decode_kernel", "pa_host_staging_size", "pa_host_staging_offsets",
           "pa_decode_host", "pa_prefill", "pa_decode_launches")
PA_STATIC_WORKSPACE_BYTES = 16 << 20


class PaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class Params(ctypes.Structure):
    """Mirror of ``pa_params_t``."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("max_seq_len", ctypes.c_int32),
        ("partition_size", ctypes.c_int32),
        ("v1_max_seq_len", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


class PrefillParams(ctypes.Structure):
    """Mirror of ``pa_prefill_params_t``."""
    _fields_ = [
        ("num_seqs", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("total_tokens", ctypes.c_int32),
        ("max_query_len", ctypes.c_int32),
        ("max_ctx_len", ctypes.c_int32),
        ("kv_dtype", ctypes.c_int32),
        ("out_dtype", ctypes.c_int32),
        ("scale", ctypes.c_float),
        ("flags", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded ``libpa.so``; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "`python -m paged_attention_decode_v2_gb300.build` (there is no fallback)")
            L = ctypes.CDLL(LIB_PATH)
            P = ctypes.c_void_p
            PP = ctypes.POINTER(Params)
            L.pa_workspace_size.argtypes = [PP]
            L.pa_workspace_size.restype = ctypes.c_size_t
            L.pa_decode_v1.argtypes = [PP, P, P, P, P, P, P, P]
            L.pa_decode_v1.restype = ctypes.c_int
            L.pa_decode_v2.argtypes = [PP, P, P, P, P, P, P, ctypes.c_size_t, P, P]
            L.pa_decode_v2.restype = ctypes.c_int
            L.pa_decode_v2_partitions.argtypes = [PP, P, P, P, P, P, P, ctypes.c_size_t, P]
            L.pa_decode_v2_partitions.restype = ctypes.c_int
            L.pa_decode_v2_reduce.argtypes = [PP, P, P, ctypes.c_size_t, P, P]
            L.pa_decode_v2_reduce.restype = ctypes.c_int
            L.pa_decode.argtypes = [PP, P, P, P, P, P, P, ctypes.c_size_t, P, P]
            L.pa_decode.restype = ctypes.c_int
            L.pa_decode_kernel.argtypes = [PP]
            L.pa_decode_kernel.restype = ctypes.c_int
            L.pa_decode_launches.argtypes = [PP]
            L.pa_decode_launches.restype = ctypes.c_int
            L.pa_decode_path.argtypes = [PP]
            L.pa_decode_path.restype = ctypes.c_int
            L.pa_status_string.argtypes = [ctypes.c_int]
            L.pa_status_string.restype = ctypes.c_char_p
            L.pa_workspace_init.argtypes = [P, ctypes.c_size_t, P]
            L.pa_workspace_init.restype = ctypes.c_int
            L.pa_read_device_status.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.c_int, P]
            L.pa_read_device_status.restype = ctypes.c_int
            L.pa_version.restype = ctypes.c_int
            L.pa_decode_v2_static.argtypes = [PP, P, P, P, P, P, P, P]
            L.pa_decode_v2_static.restype = ctypes.c_int
            L.pa_host_staging_size.argtypes = [PP]
            L.pa_host_staging_size.restype = ctypes.c_size_t
            L.pa_host_staging_offsets.argtypes = [PP, ctypes.POINTER(ctypes.c_size_t)]
            L.pa_host_staging_offsets.restype = ctypes.c_int
            L.pa_decode_host.argtypes = [PP, P, P, P, P, P, P, ctypes.c_size_t, P, ctypes.c_size_t,
                                         P, P]
            L.pa_decode_host.restype = ctypes.c_int
            L.pa_prefill.argtypes = [ctypes.POINTER(PrefillParams), P, P, P, P, P, P, P, P, P, P]
            L.pa_prefill.restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _dtype_code(dtype) -> int:
    import torch
    codes = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16}
    if dtype not in codes:
        raise PaError(PA_ERR_UNSUPPORTED, f"dtype {dtype}")
    return codes[dtype]


def cache_dims(k_cache, split_x: bool = False):
    """(num_blocks, num_kv_heads, block_size, head_dim) of a key cache in the
    standard [blocks, kv_heads, block_size, head_dim] layout, or (split_x) in
    the split-x layout [blocks, kv_heads, head_dim / x, block_size, x]."""
    if split_x:
        if k_cache.dim() != 5:
            raise PaError(PA_ERR_INVALID_ARG, "split-x k_cache must be 5-D")
        nb, hkv, dx, bs, x = k_cache.shape
        return nb, hkv, bs, dx * x
    if k_cache.dim() != 4:
        raise PaError(PA_ERR_INVALID_ARG, "k_cache must be 4-D")
    return tuple(k_cache.shape)


def make_params(q, k_cache, block_tables, *, max_seq_len: int, scale: float,
                partition_size: int = 512, out_dtype=None,
                v1_max_seq_len: int = DEFAULT_V1_MAX_SEQ_LEN, portable: bool = False,
                flags: int = 0, split_x: bool = False) -> Params:
    """Fill a :class:`Params` from tensor shapes (no device access)."""
    num_seqs, num_heads, head_dim = q.shape
    num_blocks, num_kv_heads, block_size, d2 = cache_dims(k_cache, split_x)
    if d2 != head_dim:
        raise PaError(PA_ERR_INVALID_ARG, "q and k_cache head_dim differ")
    return Params(num_seqs, num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  block_tables.shape[1], int(max_seq_len), int(partition_size),
                  int(v1_max_seq_len), _dtype_code(k_cache.dtype),
                  _dtype_code(out_dtype if out_dtype is not None else q.dtype), float(scale),
                  (PA_FLAG_PORTABLE if portable else 0) | (PA_FLAG_SPLIT_X if split_x else 0) |
                  int(flags))


def workspace_size(params: Params) -> int:
    return int(lib().pa_workspace_size(ctypes.byref(params)))


def decode_path(params: Params) -> int:
    return int(lib().pa_decode_path(ctypes.byref(params)))


def decode_kernel(params: Params) -> int:
    """2: tensor-core kernels, 1: CUDA-core kernels, 0: invalid parameters."""
    return int(lib().pa_decode_kernel(ctypes.byref(params)))


def decode_launches(params: Params) -> int:
    """Kernel launches one ``pa_decode`` call makes (1 or 2; 0 if invalid)."""
    return int(lib().pa_decode_launches(ctypes.byref(params)))


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _check_inputs(q, k_cache, v_cache, block_tables, seq_lens, out, split_x=False):
    import torch
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("seq_lens", seq_lens), ("out", out)):
        if not t.is_cuda:
            raise PaError(PA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise PaError(PA_ERR_INVALID_ARG, f"{name} must be contiguous")
    if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
        raise PaError(PA_ERR_INVALID_ARG, "block_tables and seq_lens must be int32")
    nb, hkv, bs, d = cache_dims(k_cache, split_x)
    v_shape = (nb, hkv, d, bs) if split_x else (nb, hkv, bs, d)
    if tuple(v_cache.shape) != v_shape or v_cache.dtype != k_cache.dtype or q.dtype != k_cache.dtype:
        raise PaError(PA_ERR_INVALID_ARG, "q, k_cache and v_cache must agree in dtype/shape")
    if tuple(out.shape) != tuple(q.shape):
        raise PaError(PA_ERR_INVALID_ARG, "out must have q's shape")


def _params_for(q, k_cache, block_tables, out, max_seq_len, scale, partition_size,
                v1_max_seq_len, portable, flags=0, split_x=False):
    return make_params(q, k_cache, block_tables, max_seq_len=max_seq_len, scale=scale,
                       partition_size=partition_size, out_dtype=out.dtype,
                       v1_max_seq_len=v1_max_seq_len, portable=portable, flags=flags,
                       split_x=split_x)


def decode_v1(q, k_cache, v_cache, block_tables, seq_lens, out, *, max_seq_len: int,
              scale: float, portable: bool = False, split_x: bool = False, flags: int = 0,
              stream=None):
    """``pa_decode_v1``: single pass per (sequence, KV head), into ``out``.
    ``split_x``: the caches are in the split-x layout (``PA_FLAG_SPLIT_X``);
    ``flags``: further ``PA_FLAG_*`` bits."""
    _check_inputs(q, k_cache, v_cache, block_tables, seq_lens, out, split_x)
    p = _params_for(q, k_cache, block_tables, out, max_seq_len, scale, 512,
                    DEFAULT_V1_MAX_SEQ_LEN, portable, flags, split_x)
    st = lib().pa_decode_v1(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                            _ptr(block_tables), _ptr(seq_lens), _ptr(out), _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v1")
    return out


def decode_v2(q, k_cache, v_cache, block_tables, seq_lens, out, workspace, *, max_seq_len: int,
              scale: float, partition_size: int = 512, portable: bool = False, stream=None,
              flags: int = 0, split_x: bool = False):
    """``pa_decode_v2``: split-KV pass 1 + log-sum-exp reduce, into ``out``.

    ``workspace`` is a CUDA uint8 tensor of at least :func:`workspace_size`
    bytes, allocated once and reused.
    """
    _check_inputs(q, k_cache, v_cache, block_tables, seq_lens, out, split_x)
    p = _params_for(q, k_cache, block_tables, out, max_seq_len, scale, partition_size,
                    DEFAULT_V1_MAX_SEQ_LEN, portable, flags, split_x)
    st = lib().pa_decode_v2(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                            _ptr(block_tables), _ptr(seq_lens), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _ptr(out),
                            _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2")
    return out


def decode_v2_partitions(q, k_cache, v_cache, block_tables, seq_lens, workspace, *,
                         max_seq_len: int, scale: float, partition_size: int = 512,
                         out_dtype=None, portable: bool = False, split_x: bool = False,
                         stream=None):
    """``pa_decode_v2_partitions``: V2 pass 1 only (fills the workspace)."""
    p = make_params(q, k_cache, block_tables, max_seq_len=max_seq_len, scale=scale,
                    partition_size=partition_size, out_dtype=out_dtype, portable=portable,
                    split_x=split_x)
    st = lib().pa_decode_v2_partitions(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                       _ptr(block_tables), _ptr(seq_lens), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_partitions")


def decode_v2_reduce(params: Params, seq_lens, workspace, out, stream=None):
    """``pa_decode_v2_reduce``: V2 pass 2 only (workspace -> out)."""
    st = lib().pa_decode_v2_reduce(ctypes.byref(params), _ptr(seq_lens), _ptr(workspace),
                                   workspace.numel() * workspace.element_size(), _ptr(out),
                                   _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_reduce")
    return out


def decode(q, k_cache, v_cache, block_tables, seq_lens, out, workspace=None, *,
           max_seq_len: int, scale: float, partition_size: int = 512,
           v1_max_seq_len: int = DEFAULT_V1_MAX_SEQ_LEN, portable: bool = False,
           split_x: bool = False, stream=None):
    """``pa_decode``: V2 when ``max_seq_len > v1_max_seq_len``, else V1."""
    _check_inputs(q, k_cache, v_cache, block_tables, seq_lens, out, split_x)
    p = _params_for(q, k_cache, block_tables, out, max_seq_len, scale, partition_size,
                    v1_max_seq_len, portable, split_x=split_x)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().pa_decode(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                         _ptr(block_tables), _ptr(seq_lens), _ptr(workspace), nbytes, _ptr(out),
                         _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode")
    return out


def decode_v2_static(q, k_cache, v_cache, block_tables, seq_lens, out, *, max_seq_len: int,
                     scale: float, partition_size: int = 512, portable: bool = False,
                     stream=None):
    """``pa_decode_v2_static``: V2 with the library's own fixed 16 MiB device
    workspace, for callers that cannot allocate one.  Calls on a device share
    that workspace, so calls that overlap on the GPU race."""
    _check_inputs(q, k_cache, v_cache, block_tables, seq_lens, out)
    p = _params_for(q, k_cache, block_tables, out, max_seq_len, scale, partition_size,
                    DEFAULT_V1_MAX_SEQ_LEN, portable)
    st = lib().pa_decode_v2_static(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                                   _ptr(block_tables), _ptr(seq_lens), _ptr(out), _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode_v2_static")
    return out


def host_staging_size(params: Params) -> int:
    return int(lib().pa_host_staging_size(ctypes.byref(params)))


def alloc_host_staging(params: Params, device=None):
    """A CUDA uint8 tensor of :func:`host_staging_size` bytes for
    :func:`decode_host` (allocated by torch, reused across calls)."""
    import torch
    n = host_staging_size(params)
    if n == 0:
        raise PaError(PA_ERR_INVALID_ARG, "pa_host_staging_size")
    return torch.empty(n, dtype=torch.uint8, device=device or "cuda")


def host_staging_offsets(params: Params):
    """``pa_host_staging_offsets``: byte offsets of q, block_tables, seq_lens
    and out in the staging layout, and its total size."""
    arr = (ctypes.c_size_t * 5)()
    st = lib().pa_host_staging_offsets(ctypes.byref(params), arr)
    if st != PA_OK:
        raise PaError(st, "pa_host_staging_offsets")
    return tuple(int(x) for x in arr)


def alloc_host_mirror(params: Params, q_dtype, num_seqs: int, num_heads: int, head_dim: int,
                      max_blocks_per_seq: int):
    """A pinned host buffer with the staging layout, and CPU tensors viewing
    its q, block_tables and seq_lens regions.  Inputs written there are moved
    by :func:`decode_host` in one copy."""
    import torch
    off = host_staging_offsets(params)
    buf = torch.zeros(off[4], dtype=torch.uint8).pin_memory()
    esz = torch.tensor([], dtype=q_dtype).element_size()
    nq = num_seqs * num_heads * head_dim
    q = buf[:nq * esz].view(q_dtype).view(num_seqs, num_heads, head_dim)
    bt = buf[off[1]:off[1] + num_seqs * max_blocks_per_seq * 4].view(torch.int32)
    sl = buf[off[2]:off[2] + num_seqs * 4].view(torch.int32)
    return buf, q, bt.view(num_seqs, max_blocks_per_seq), sl


def decode_host(q, k_cache, v_cache, block_tables, seq_lens, out, workspace, staging, *,
                max_seq_len: int = 0, scale: float = 0.0, partition_size: int = 512,
                v1_max_seq_len: int = DEFAULT_V1_MAX_SEQ_LEN, portable: bool = False,
                params: Params | None = None, stream=None):
    """``pa_decode_host``: the decode step with q, block_tables, seq_lens and
    ``out`` in HOST memory (CPU tensors; pinned ones make the copies
    asynchronous), the caches and ``workspace`` (None for V1) and
    ``staging`` (see :func:`alloc_host_staging`) on the device.  Returns when
    ``out`` holds the result.  ``params`` (from :func:`make_params`) may be
    passed to reuse one description across steps."""
    if params is None:
        import torch
        for name, t in (("q", q), ("block_tables", block_tables), ("seq_lens", seq_lens),
                        ("out", out)):
            if t.is_cuda or not t.is_contiguous():
                raise PaError(PA_ERR_INVALID_ARG, f"{name} must be a contiguous host tensor")
        for name, t in (("k_cache", k_cache), ("v_cache", v_cache)):
            if not t.is_cuda or not t.is_contiguous():
                raise PaError(PA_ERR_INVALID_ARG, f"{name} must be a contiguous CUDA tensor")
        if block_tables.dtype != torch.int32 or seq_lens.dtype != torch.int32:
            raise PaError(PA_ERR_INVALID_ARG, "block_tables and seq_lens must be int32")
        if tuple(out.shape) != tuple(q.shape):
            raise PaError(PA_ERR_INVALID_ARG, "out must have q's shape")
        params = _params_for(q, k_cache, block_tables, out, max_seq_len, scale, partition_size,
                             v1_max_seq_len, portable)
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().pa_decode_host(ctypes.byref(params), _ptr(q), _ptr(k_cache), _ptr(v_cache),
                              _ptr(block_tables), _ptr(seq_lens), _ptr(workspace), nbytes,
                              _ptr(staging), staging.numel(), _ptr(out), _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_decode_host")
    return out


def alloc_workspace(params: Params, device=None):
    """A CUDA uint8 tensor sized for ``params`` (allocated by torch), with its
    control block initialised by :func:`workspace_init`."""
    import torch
    n = workspace_size(params)
    if n == 0:
        raise PaError(PA_ERR_INVALID_ARG, "pa_workspace_size")
    ws = torch.empty(n, dtype=torch.uint8, device=device or "cuda")
    workspace_init(ws)
    return ws


def workspace_init(workspace, stream=None):
    st = lib().pa_workspace_init(_ptr(workspace), workspace.numel(), _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_workspace_init")


def read_device_status(workspace, clear: bool = True, stream=None) -> int:
    """The device status word (waits for the stream)."""
    v = ctypes.c_int32(0)
    st = lib().pa_read_device_status(_ptr(workspace), ctypes.byref(v), int(clear),
                                     _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_read_device_status")
    return int(v.value)


def version() -> int:
    return int(lib().pa_version())


def make_prefill_params(q, k_cache, block_tables, *, max_query_len: int, max_ctx_len: int,
                        scale: float, out_dtype=None, flags: int = 0) -> PrefillParams:
    """Fill a :class:`PrefillParams` from tensor shapes (no device access)."""
    total_tokens, num_heads, head_dim = q.shape
    num_blocks, num_kv_heads, block_size, d2 = cache_dims(k_cache)
    if d2 != head_dim:
        raise PaError(PA_ERR_INVALID_ARG, "q and k_cache head_dim differ")
    return PrefillParams(block_tables.shape[0], num_heads, num_kv_heads, head_dim, block_size,
                         num_blocks, block_tables.shape[1], total_tokens, int(max_query_len),
                         int(max_ctx_len), _dtype_code(k_cache.dtype),
                         _dtype_code(out_dtype if out_dtype is not None else q.dtype),
                         float(scale), int(flags))


def prefill(q, k, v, k_cache, v_cache, block_tables, query_start, ctx_lens, out, *,
            max_query_len: int, max_ctx_len: int, scale: float, flags: int = 0, stream=None):
    """``pa_prefill``: paged prefix prefill of a chunk of new tokens per
    sequence.  ``q`` [T, Hq, D], ``k`` / ``v`` [T, Hkv, D], the caches
    [blocks, Hkv, BS, D], ``block_tables`` [B, max_blocks], ``query_start``
    [B + 1], ``ctx_lens`` [B], ``out`` [T, Hq, D] (CUDA tensors)."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("k_cache", k_cache), ("v_cache", v_cache),
                    ("block_tables", block_tables), ("query_start", query_start),
                    ("ctx_lens", ctx_lens), ("out", out)):
        if not t.is_cuda:
            raise PaError(PA_ERR_INVALID_ARG, f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise PaError(PA_ERR_INVALID_ARG, f"{name} must be contiguous")
    for t in (block_tables, query_start, ctx_lens):
        if t.dtype != torch.int32:
            raise PaError(PA_ERR_INVALID_ARG, "block_tables, query_start and ctx_lens must be int32")
    T, hq, d = q.shape
    nb, hkv, bs, d2 = cache_dims(k_cache)
    if (tuple(k.shape) != (T, hkv, d) or tuple(v.shape) != (T, hkv, d) or d2 != d or
            tuple(v_cache.shape) != tuple(k_cache.shape) or tuple(out.shape) != tuple(q.shape)):
        raise PaError(PA_ERR_INVALID_ARG, "prefill tensor shapes disagree")
    if not (q.dtype == k.dtype == v.dtype == k_cache.dtype == v_cache.dtype):
        raise PaError(PA_ERR_INVALID_ARG, "q, k, v and the caches must share one dtype")
    B = block_tables.shape[0]
    if tuple(query_start.shape) != (B + 1,) or tuple(ctx_lens.shape) != (B,):
        raise PaError(PA_ERR_INVALID_ARG, "query_start must be [B + 1] and ctx_lens [B]")
    params = make_prefill_params(q, k_cache, block_tables, max_query_len=max_query_len,
                                 max_ctx_len=max_ctx_len, scale=scale, out_dtype=out.dtype,
                                 flags=flags)
    st = lib().pa_prefill(ctypes.byref(params), _ptr(q), _ptr(k), _ptr(v), _ptr(k_cache),
                          _ptr(v_cache), _ptr(block_tables), _ptr(query_start), _ptr(ctx_lens),
                          _ptr(out), _stream(stream))
    if st != PA_OK:
        raise PaError(st, "pa_prefill")
