"""pa_decode_v2_static, the decode entry point that allocates nothing.

Some callers cannot allocate device memory where they decode (a plugin of a
host runtime that owns every device allocation, a C program without an
allocator, a real-time loop that must not stall on one).  For them
pa_decode_v2_static runs V2 with a fixed workspace the library keeps in
device memory.  This file checks, through the C ABI, that on two calls in a
row (the second call sees whatever the first left in the shared array) its
output matches the float64 oracle on NaN-poisoned inputs, and pa_decode_v2
with a caller-provided workspace, within the parity tolerance; that a block
id outside the pool turns exactly that sequence's rows into NaN; and that
oversized parameters are refused before anything runs.

The file is named to be collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import paged_attention_decode_v2_gb300 as pa
from paged_attention_decode_v2_gb300 import workloads as wl
from gpu_helpers import TOL, max_err
from oracle_pins import problem

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


def test_static_workspace_matches_oracle_and_decode_v2_on_two_calls():
    from paged_attention_decode_v2_gb300 import build
    build.build()
    assert torch.cuda.is_available()
    # two different batches: the second call runs on what the first left behind
    batches = [
        (wl.make(wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=6, max_len=20000), poison=True),
         512),
        (wl.make(wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=12345), poison=True), 1024),
    ]
    for bc, P in batches:
        ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens,
                            bc.scale)
        b = bc.to("cuda")
        want = _reference_v2(b, P)
        got = torch.full(tuple(b.q.shape), float("nan"), dtype=torch.float32, device="cuda")
        assert _call_static(b, got, P) == pa.PA_OK
        torch.cuda.synchronize()
        g = got.double().cpu().numpy()
        assert np.all(np.isfinite(g))
        err = max_err(g, ref)
        assert err <= TOL[b.q.dtype], f"static workspace differs from the oracle by {err}"
        err = max_err(g, want.double().cpu().numpy())
        assert err <= TOL[b.q.dtype], f"static workspace differs from decode_v2 by {err}"


def test_static_workspace_bad_block_id_gives_nan_rows():
    """A block id outside the pool makes exactly that sequence's rows NaN
    (the call reports no device status); the other rows match the oracle."""
    lens = (900, 700, 1300)
    good = problem(dtype=torch.bfloat16, lens=lens, Hq=8, Hkv=2, D=128, BS=16, seed=31)
    ref = oracle.decode(good.q, good.k_cache, good.v_cache, good.block_tables, good.seq_lens,
                        good.scale)
    bad = problem(dtype=torch.bfloat16, lens=lens, Hq=8, Hkv=2, D=128, BS=16, seed=31)
    bad.block_tables[1, 20] = bad.k_cache.shape[0] + 3      # token 320 of sequence 1
    b = bad.to("cuda")
    got = torch.zeros(tuple(b.q.shape), dtype=torch.float32, device="cuda")
    assert _call_static(b, got, 256) == pa.PA_OK
    torch.cuda.synchronize()
    g = got.double().cpu().numpy()
    assert np.all(np.isnan(g[1]))
    for s in (0, 2):
        assert np.all(np.isfinite(g[s]))
        assert max_err(g[s], ref[s]) <= TOL[torch.bfloat16]


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
