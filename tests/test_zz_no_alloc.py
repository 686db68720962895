"""pa_decode_v2_static, the decode entry point that allocates nothing.

Some callers cannot allocate device memory where they decode (a plugin of a
host runtime that owns every device allocation, a C program without an
allocator, a real-time loop that must not stall on one).  For them
pa_decode_v2_static runs V2 with a fixed workspace the library keeps in
device memory.  This file checks, through the C ABI, that it gives the same
output as pa_decode_v2 with a caller-provided workspace, on two calls in a
row (the second call sees whatever the first left in the shared array), and
that oversized parameters are refused before anything runs.

The file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import pytest
import torch

import paged_attention_decode_v2_gb300 as pa
from paged_attention_decode_v2_gb300 import workloads as wl
from gpu_helpers import TOL, max_err

pytestmark = pytest.mark.gpu


def _call_static(b, out, P):
    p = pa.make_params(b.q, b.k_cache, b.block_tables, max_seq_len=b.max_seq_len, scale=b.scale,
                       partition_size=P, out_dtype=out.dtype)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return pa.lib().pa_decode_v2_static(
        ctypes.byref(p), ctypes.c_void_p(b.q.data_ptr()), ctypes.c_void_p(b.k_cache.data_ptr()),
        ctypes.c_void_p(b.v_cache.data_ptr()), ctypes.c_void_p(b.block_tables.data_ptr()),
        ctypes.c_void_p(b.seq_lens.data_ptr()), ctypes.c_void_p(out.data_ptr()), stream)


def _reference_v2(b, P):
    params = pa.make_params(b.q, b.k_cache, b.block_tables, max_seq_len=b.max_seq_len,
                            scale=b.scale, partition_size=P, out_dtype=torch.float32)
    ws = pa.alloc_workspace(params)
    out = torch.empty(tuple(b.q.shape), dtype=torch.float32, device="cuda")
    pa.decode_v2(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, out, ws,
                 max_seq_len=b.max_seq_len, scale=b.scale, partition_size=P)
    return out


def test_static_workspace_matches_decode_v2_on_two_calls():
    from paged_attention_decode_v2_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    # two different batches: the second call runs on what the first left behind
    batches = [
        (wl.make(wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=6, max_len=20000), device="cuda",
                 poison=True), 512),
        (wl.make(wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=12345), device="cuda", poison=True),
         1024),
    ]
    for b, P in batches:
        want = _reference_v2(b, P)
        got = torch.full(tuple(b.q.shape), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(b, got, P) == pa.PA_OK
        torch.cuda.synchronize()
        assert torch.isfinite(got).all().item()
        err = max_err(got.double().cpu().numpy(), want.double().cpu().numpy())
        assert err <= TOL[b.q.dtype], f"static workspace differs from decode_v2 by {err}"


def test_static_workspace_rejects_oversized_parameters():
    # 256 sequences x 32 heads x 256 partitions x head_dim 128 needs about
    # 1 GiB of workspace: refused by a host check, nothing is enqueued
    p = pa.Params(256, 32, 8, 128, 32, 40000, 4096, 131072, 512, 0, pa.PA_BF16, pa.PA_F32,
                  0.088, 0)
    assert pa.workspace_size(p) > pa.PA_STATIC_WORKSPACE_BYTES
    V = ctypes.c_void_p
    st = pa.lib().pa_decode_v2_static(ctypes.byref(p), V(256), V(256), V(256), V(256), V(256),
                                      V(256), V(0))
    assert st == pa.PA_ERR_WORKSPACE_TOO_SMALL
