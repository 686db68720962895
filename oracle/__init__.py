"""Float64 CPU oracle for paged single-token decode attention and paged
prefix prefill.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product library
never imports this package, and this package imports nothing from it.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision); this
module compiles it with gcc and marshals arrays through ctypes.  Inputs are
the exact element bits the GPU path reads (float32, bfloat16 or float16
torch CPU tensors); the C code widens them to double itself.

Sources (commit pages of the project "project_6"):
  * commit 4eb83a7e "qwen3_6_scripts", paragraph "Implementation
    (paged_attention_v2_pytorch.py)": Phase 1 / Phase 2 of the V2 split-KV
    scheme, followed step by step by :func:`decode_partitioned`;
  * commit 4eb83a7e "qwen3_6_scripts", paragraph "V1 paged_attention
    (decode <= 8192)": V1 is checked against plain ("manual") attention,
    which is :func:`decode`;
  * commit 4eb83a7e "qwen3_6_scripts", paragraph "Hardware testing
    confirmed": the [blocks, kv_heads, block_size, head_dim] cache layout;
  * commit 1a4e1005 "paged_attn.py", opening paragraph, and commit 4eb83a7e
    "qwen3_6_scripts", paragraphs on the prefix attention's pre-allocated
    buffers, "Complete rewrite of qwen3_6_scripts/paged_attn.py" (item 1)
    and "Prefill (flash_attn_func)": prefill as online softmax over key
    tiles, a context phase from the paged cache then a causal phase over the
    chunk's own tokens -- :func:`prefill` is the plain definition,
    :func:`prefill_tiled` the tiled algorithm.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "libpa_oracle.so")
_lock = threading.Lock()

_DTYPE_CODE = {torch.float32: 0, torch.bfloat16: 1, torch.float16: 2}


class _Shape(ctypes.Structure):
    _fields_ = [
        ("dtype", ctypes.c_int32),
        ("num_seqs", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
        ("num_blocks", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32),
        ("scale", ctypes.c_double),
    ]


def source() -> str:
    """Path of the oracle's C source."""
    return _SRC


def build(force: bool = False, src: str | None = None, out: str | None = None) -> str:
    """Compile ``pa_oracle.c`` into a shared library (gcc, -O2, OpenMP).

    ``src`` and ``out`` exist so the test suite can compile deliberately
    broken copies of the oracle (in a temporary directory) and check that its
    pins catch them; the default build uses neither.
    """
    src = src or _SRC
    target = out or _LIB
    if (not force and src == _SRC and os.path.exists(target)
            and os.path.getmtime(target) >= os.path.getmtime(_SRC)):
        return target
    tmp = target + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, target)
    return target


def _prep(q, k_cache, v_cache, block_tables, seq_lens, scale):
    for name, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache)):
        if t.device.type != "cpu":
            raise ValueError(f"oracle: {name} must be a CPU tensor")
    if not (q.dtype == k_cache.dtype == v_cache.dtype) or q.dtype not in _DTYPE_CODE:
        raise ValueError("oracle: q, k_cache and v_cache must share one of f32/bf16/f16")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or q.dim() != 3:
        raise ValueError("oracle: q [B,Hq,D], caches [blocks, kv_heads, block_size, D]")
    nb, hkv, bs, d = k_cache.shape
    b, hq, dq = q.shape
    if dq != d:
        raise ValueError("oracle: head_dim mismatch")
    bt = block_tables.cpu().to(torch.int32).contiguous()
    sl = seq_lens.cpu().to(torch.int32).contiguous()
    if bt.dim() != 2 or bt.shape[0] != b or sl.shape != (b,):
        raise ValueError("oracle: block_tables [B, max_blocks], seq_lens [B]")
    shape = _Shape(_DTYPE_CODE[q.dtype], b, hq, hkv, d, bs, nb, bt.shape[1], float(scale))
    keep = [q.contiguous(), k_cache.contiguous(), v_cache.contiguous(), bt, sl]
    return shape, keep


def _prep_prefill(q, k_new, v_new, k_cache, v_cache, block_tables, query_start, ctx_lens,
                  scale):
    for name, t in (("q", q), ("k_new", k_new), ("v_new", v_new), ("k_cache", k_cache),
                    ("v_cache", v_cache)):
        if t.device.type != "cpu":
            raise ValueError(f"oracle: {name} must be a CPU tensor")
        if t.dtype != q.dtype:
            raise ValueError("oracle: q, k_new, v_new and the caches must share one dtype")
    if q.dtype not in _DTYPE_CODE:
        raise ValueError("oracle: dtype must be f32, bf16 or f16")
    if k_cache.dim() != 4 or v_cache.shape != k_cache.shape or q.dim() != 3:
        raise ValueError("oracle: q [T,Hq,D], caches [blocks, kv_heads, block_size, D]")
    nb, hkv, bs, d = k_cache.shape
    T, hq, dq = q.shape
    if dq != d or k_new.shape != (T, hkv, d) or v_new.shape != (T, hkv, d):
        raise ValueError("oracle: k_new / v_new must be [T, Hkv, D]")
    bt = block_tables.cpu().to(torch.int32).contiguous()
    qs = query_start.cpu().to(torch.int32).contiguous()
    cl = ctx_lens.cpu().to(torch.int32).contiguous()
    B = cl.shape[0]
    if bt.dim() != 2 or bt.shape[0] != B or qs.shape != (B + 1,):
        raise ValueError("oracle: block_tables [B, max_blocks], query_start [B+1], ctx_lens [B]")
    shape = _Shape(_DTYPE_CODE[q.dtype], B, hq, hkv, d, bs, nb, bt.shape[1], float(scale))
    keep = [q.contiguous(), k_new.contiguous(), v_new.contiguous(), k_cache.contiguous(),
            v_cache.contiguous(), bt, qs, cl]
    return shape, T, keep


def _check(rc: int) -> None:
    if rc == -2:
        raise ValueError("oracle: block table entry outside the pool")
    if rc != 0:
        raise ValueError(f"oracle: bad arguments (code {rc})")


class Oracle:
    """ctypes handle on one build of ``pa_oracle.c``."""

    def __init__(self, path: str):
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        lib.pa_oracle_decode.argtypes = [ctypes.POINTER(_Shape), P, P, P, P, P, P,
                                         ctypes.c_int64, P]
        lib.pa_oracle_decode.restype = ctypes.c_int
        lib.pa_oracle_decode_partitioned.argtypes = [
            ctypes.POINTER(_Shape), P, P, P, P, P, ctypes.c_int32, ctypes.c_int32,
            P, P, P, P]
        lib.pa_oracle_decode_partitioned.restype = ctypes.c_int
        lib.pa_oracle_prefill.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int64, P, P, P, P,
                                          P, P, P, P, P, ctypes.c_int64, P]
        lib.pa_oracle_prefill.restype = ctypes.c_int
        lib.pa_oracle_prefill_tiled.argtypes = [ctypes.POINTER(_Shape), ctypes.c_int64, P, P,
                                                P, P, P, P, P, P, ctypes.c_int32, P]
        lib.pa_oracle_prefill_tiled.restype = ctypes.c_int
        lib.pa_oracle_max_threads.restype = ctypes.c_int
        lib.pa_oracle_set_threads.argtypes = [ctypes.c_int]
        self.lib = lib
        self.path = path

    def max_threads(self) -> int:
        return self.lib.pa_oracle_max_threads()

    def set_threads(self, n: int) -> None:
        self.lib.pa_oracle_set_threads(int(n))

    def decode(self, q, k_cache, v_cache, block_tables, seq_lens, scale, rows=None):
        """Plain softmax attention of each query row over its paged keys/values.

        Returns float64 ``[B, Hq, D]``; with ``rows`` (flat ``b*Hq + h``
        indices) returns ``[len(rows), D]`` for those rows only.
        """
        shape, keep = _prep(q, k_cache, v_cache, block_tables, seq_lens, scale)
        qc, kc, vc, bt, sl = keep
        d = shape.head_dim
        if rows is None:
            out = np.empty((shape.num_seqs, shape.num_heads, d), dtype=np.float64)
            rows_arr, nrows, rows_ptr = None, 0, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            nrows = rows_arr.size
            rows_ptr = rows_arr.ctypes.data
            out = np.empty((nrows, d), dtype=np.float64)
        rc = self.lib.pa_oracle_decode(ctypes.byref(shape), qc.data_ptr(), kc.data_ptr(),
                                       vc.data_ptr(), bt.data_ptr(), sl.data_ptr(), rows_ptr,
                                       nrows, out.ctypes.data)
        _check(rc)
        return out

    def decode_partitioned(self, q, k_cache, v_cache, block_tables, seq_lens, scale,
                           partition_size, max_partitions=None):
        """The V2 two-phase scheme in double.

        Returns ``(out, max_logits, exp_sums, tmp_out)`` with shapes
        ``[B,Hq,D]``, ``[B,Hq,NP]``, ``[B,Hq,NP]`` and ``[B,Hq,NP,D]``;
        partitions a sequence does not have are NaN.
        """
        shape, keep = _prep(q, k_cache, v_cache, block_tables, seq_lens, scale)
        qc, kc, vc, bt, sl = keep
        p = int(partition_size)
        if max_partitions is None:
            mx = int(sl.max().item()) if sl.numel() else 0
            max_partitions = max(1, -(-mx // p))
        b, hq, d = shape.num_seqs, shape.num_heads, shape.head_dim
        np_ = int(max_partitions)
        out = np.empty((b, hq, d), dtype=np.float64)
        ml = np.full((b, hq, np_), np.nan)
        es = np.full((b, hq, np_), np.nan)
        to = np.full((b, hq, np_, d), np.nan)
        rc = self.lib.pa_oracle_decode_partitioned(
            ctypes.byref(shape), qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), bt.data_ptr(),
            sl.data_ptr(), p, np_, ml.ctypes.data, es.ctypes.data, to.ctypes.data,
            out.ctypes.data)
        _check(rc)
        return out, ml, es, to


    def prefill(self, q, k_new, v_new, k_cache, v_cache, block_tables, query_start, ctx_lens,
                scale, rows=None):
        """Paged prefix prefill by the plain definition: query row (t, h) of
        sequence b (query_start[b] <= t < query_start[b+1], i = t -
        query_start[b]) attends to the sequence's ctx_lens[b] cached tokens
        and to its new tokens 0..i (k_new / v_new rows query_start[b]..t).

        Returns float64 ``[T, Hq, D]``; with ``rows`` (flat ``t*Hq + h``
        indices) returns ``[len(rows), D]``.
        """
        shape, T, keep = _prep_prefill(q, k_new, v_new, k_cache, v_cache, block_tables,
                                       query_start, ctx_lens, scale)
        qc, kn, vn, kc, vc, bt, qs, cl = keep
        d = shape.head_dim
        if rows is None:
            out = np.empty((T, shape.num_heads, d), dtype=np.float64)
            rows_arr, nrows, rows_ptr = None, 0, None
        else:
            rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
            nrows = rows_arr.size
            rows_ptr = rows_arr.ctypes.data
            out = np.empty((nrows, d), dtype=np.float64)
        rc = self.lib.pa_oracle_prefill(ctypes.byref(shape), T, qc.data_ptr(), kn.data_ptr(),
                                        vn.data_ptr(), kc.data_ptr(), vc.data_ptr(),
                                        bt.data_ptr(), qs.data_ptr(), cl.data_ptr(), rows_ptr,
                                        nrows, out.ctypes.data)
        _check(rc)
        return out

    def prefill_tiled(self, q, k_new, v_new, k_cache, v_cache, block_tables, query_start,
                      ctx_lens, scale, tile):
        """The pages' tiled online-softmax prefill (context tiles, then chunk
        tiles), in double; ``[T, Hq, D]``."""
        shape, T, keep = _prep_prefill(q, k_new, v_new, k_cache, v_cache, block_tables,
                                       query_start, ctx_lens, scale)
        qc, kn, vn, kc, vc, bt, qs, cl = keep
        out = np.empty((T, shape.num_heads, shape.head_dim), dtype=np.float64)
        rc = self.lib.pa_oracle_prefill_tiled(ctypes.byref(shape), T, qc.data_ptr(),
                                              kn.data_ptr(), vn.data_ptr(), kc.data_ptr(),
                                              vc.data_ptr(), bt.data_ptr(), qs.data_ptr(),
                                              cl.data_ptr(), int(tile), out.ctypes.data)
        _check(rc)
        return out


_default = None


def default() -> Oracle:
    """The oracle built from the unmodified source."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def max_threads() -> int:
    """Number of OpenMP threads the oracle will use."""
    return default().max_threads()


def set_threads(n: int) -> None:
    default().set_threads(n)


def decode(q, k_cache, v_cache, block_tables, seq_lens, scale, rows=None) -> np.ndarray:
    """See :meth:`Oracle.decode`."""
    return default().decode(q, k_cache, v_cache, block_tables, seq_lens, scale, rows)


def decode_partitioned(q, k_cache, v_cache, block_tables, seq_lens, scale, partition_size,
                       max_partitions=None):
    """See :meth:`Oracle.decode_partitioned`."""
    return default().decode_partitioned(q, k_cache, v_cache, block_tables, seq_lens, scale,
                                        partition_size, max_partitions)


def prefill(q, k_new, v_new, k_cache, v_cache, block_tables, query_start, ctx_lens, scale,
            rows=None) -> np.ndarray:
    """See :meth:`Oracle.prefill`."""
    return default().prefill(q, k_new, v_new, k_cache, v_cache, block_tables, query_start,
                             ctx_lens, scale, rows)


def prefill_tiled(q, k_new, v_new, k_cache, v_cache, block_tables, query_start, ctx_lens,
                  scale, tile) -> np.ndarray:
    """See :meth:`Oracle.prefill_tiled`."""
    return default().prefill_tiled(q, k_new, v_new, k_cache, v_cache, block_tables,
                                   query_start, ctx_lens, scale, tile)
