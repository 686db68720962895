"""Failure detection on the GPU without a fault.

Every wait in the tensor-core kernel is bounded.  PA_FLAG_SELFTEST_STALL makes
the kernel wait for an event that never happens (with a ~10 ms bound): the
wait runs out, the kernel drains what it had in flight, releases its tensor
memory and returns; the host then reads PA_ERR_DEVICE_TIMEOUT from the status
word, the outputs are NaN, and the same CUDA context decodes correctly
afterwards.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_attention_decode_v2_gb300 as pa
from paged_attention_decode_v2_gb300 import workloads as wl
from gpu_helpers import MARKER, control_words

pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_reports_timeout_and_context_survives():
    from paged_attention_decode_v2_gb300 import build
    build.build()
    bc = wl.make(wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=3000), poison=True)
    bg = bc.to("cuda")
    P = 512
    params = pa.make_params(bg.q, bg.k_cache, bg.block_tables, max_seq_len=bg.max_seq_len,
                            scale=bg.scale, partition_size=P, out_dtype=torch.float32)
    assert pa.decode_kernel(params) == 2, "the self-test needs the tensor-core path"
    ws = pa.alloc_workspace(params)
    kw = dict(max_seq_len=bg.max_seq_len, scale=bg.scale, partition_size=P)

    out = torch.zeros(tuple(bg.q.shape), dtype=torch.float32, device="cuda")
    pa.decode_v2(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws,
                 flags=pa.PA_FLAG_SELFTEST_STALL, **kw)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws) == pa.PA_ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all().item()

    # the context is still usable: a normal call succeeds and is correct
    pa.decode_v2(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws, **kw)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws) == pa.PA_OK
    ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens, bc.scale)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= 2e-3


def test_one_launch_step_with_a_wait_that_runs_out():
    """The one-launch V2 step (pass 2 in the pass-1 grid) with every CTA's
    waits running out: the grid still meets at its end, the outputs are NaN,
    the status reads PA_ERR_DEVICE_TIMEOUT, the control block is ready for
    the next launch (epoch advanced, start count back at zero), and the next
    call is exact."""
    bc = wl.make(wl.scaled(wl.WORKLOADS["long_100k"], seq_len=30000), poison=True)
    bg = bc.to("cuda")
    P = 512
    params = pa.make_params(bg.q, bg.k_cache, bg.block_tables, max_seq_len=bg.max_seq_len,
                            scale=bg.scale, partition_size=P, out_dtype=torch.float32)
    assert pa.decode_launches(params) == 1
    ws = pa.alloc_workspace(params)
    kw = dict(max_seq_len=bg.max_seq_len, scale=bg.scale, partition_size=P)
    out = torch.zeros(tuple(bg.q.shape), dtype=torch.float32, device="cuda")
    pa.decode_v2(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws,
                 flags=pa.PA_FLAG_SELFTEST_STALL, **kw)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws) == pa.PA_ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all().item()
    marker, epoch, started, _, _ = control_words(ws)
    assert marker == MARKER and epoch == 1 and started == 0
    pa.decode_v2(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws, **kw)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws) == pa.PA_OK
    ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens, bc.scale)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= 2e-3


def test_prefill_wait_that_runs_out_gives_nan_and_context_survives():
    """The prefill kernel's bounded waits: with PA_FLAG_SELFTEST_STALL its
    MMA warp waits for an event that never happens, gives up after ~10 ms,
    drains and returns; the outputs are NaN and the next call is correct."""
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=(300,), new=(200,), Hq=4,
                                            Hkv=2, D=128, BS=16, seed=1))
    g = pb.to("cuda")
    out = torch.zeros(tuple(g.q.shape), dtype=torch.float32, device="cuda")
    kw = dict(max_query_len=pb.max_query_len, max_ctx_len=pb.max_ctx_len, scale=pb.scale)
    pa.prefill(g.q, g.k, g.v, g.k_cache, g.v_cache, g.block_tables, g.query_start, g.ctx_lens,
               out, flags=pa.PA_FLAG_SELFTEST_STALL, **kw)
    torch.cuda.synchronize()
    assert torch.isnan(out).all().item()
    pa.prefill(g.q, g.k, g.v, g.k_cache, g.v_cache, g.block_tables, g.query_start, g.ctx_lens,
               out, **kw)
    torch.cuda.synchronize()
    ref = oracle.prefill(pb.q, pb.k, pb.v, pb.k_cache, pb.v_cache, pb.block_tables,
                         pb.query_start, pb.ctx_lens, pb.scale)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= 4e-3


def test_split_x_wait_that_runs_out():
    """The split-x tensor-core kernel's bounded waits (PA_FLAG_SELFTEST_STALL):
    the one-launch V2 step (persistent grid, pass 2 in the same launch) and
    V1 in clusters (CTAs sharing a sequence and merging in distributed shared
    memory) both end with NaN outputs instead of hanging, V2's status word
    reads PA_ERR_DEVICE_TIMEOUT, and the next calls on the same context are
    exact."""
    from gpu_helpers import split_x_caches
    bc = wl.make(wl.scaled(wl.WORKLOADS["long_100k"], seq_len=30000), poison=True)
    bg = bc.to("cuda")
    k5, v4 = split_x_caches(bg)
    P = 512
    params = pa.make_params(bg.q, k5, bg.block_tables, max_seq_len=bg.max_seq_len,
                            scale=bg.scale, partition_size=P, out_dtype=torch.float32,
                            split_x=True)
    assert pa.decode_kernel(params) == 2 and pa.decode_launches(params) == 1
    ws = pa.alloc_workspace(params)
    kw = dict(max_seq_len=bg.max_seq_len, scale=bg.scale, split_x=True)
    ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens, bc.scale)
    out = torch.zeros(tuple(bg.q.shape), dtype=torch.float32, device="cuda")
    pa.decode_v2(bg.q, k5, v4, bg.block_tables, bg.seq_lens, out, ws, partition_size=P,
                 flags=pa.PA_FLAG_SELFTEST_STALL, **kw)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws) == pa.PA_ERR_DEVICE_TIMEOUT
    assert torch.isnan(out).all().item()
    marker, epoch, started, _, _ = control_words(ws)
    assert (marker, epoch, started) == (MARKER, 1, 0)
    pa.decode_v2(bg.q, k5, v4, bg.block_tables, bg.seq_lens, out, ws, partition_size=P, **kw)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws) == pa.PA_OK
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= 2e-3
    # V1 on one 8192-token sequence: clusters of CTAs share it
    bc = wl.make(wl.WORKLOADS["gqa_8k"], poison=True)
    bg = bc.to("cuda")
    k5, v4 = split_x_caches(bg)
    out = torch.zeros(tuple(bg.q.shape), dtype=torch.float32, device="cuda")
    kw = dict(max_seq_len=bg.max_seq_len, scale=bg.scale, split_x=True)
    pa.decode_v1(bg.q, k5, v4, bg.block_tables, bg.seq_lens, out,
                 flags=pa.PA_FLAG_SELFTEST_STALL, **kw)
    torch.cuda.synchronize()
    assert torch.isnan(out).all().item()
    pa.decode_v1(bg.q, k5, v4, bg.block_tables, bg.seq_lens, out, **kw)
    torch.cuda.synchronize()
    ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens, bc.scale)
    assert float(np.max(np.abs(out.double().cpu().numpy() - ref))) <= 2e-3
