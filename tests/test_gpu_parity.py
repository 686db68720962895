"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Tolerance (max abs error on float32 output): 2e-3 for bf16/f16 caches with
float32 accumulation, 1e-5 for float32 caches.  Inputs are NaN-poisoned
everywhere outside the batch's tokens (unused pool blocks, slots past the
last token, block-table entries past the last block are -1), and the V2
workspace is NaN-filled before each call, so reading anything the method
does not use shows up as NaN.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_attention_decode_v2_gb300 as pa
from paged_attention_decode_v2_gb300 import workloads as wl
from gpu_helpers import (MARKER, TOL, assert_close, bf16_round, control_words, max_err, run,
                         split_x_caches, workspace_views)
from oracle_pins import problem

pytestmark = pytest.mark.gpu

PATH_MODES = [("v1", False), ("v2", False), ("v1", True), ("v2", True)]


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_attention_decode_v2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _ref(batch_cpu):
    return oracle.decode(batch_cpu.q, batch_cpu.k_cache, batch_cpu.v_cache,
                         batch_cpu.block_tables, batch_cpu.seq_lens, batch_cpu.scale)


# ---------------------------------------------------------------------------
# small batches with each workload's head shapes: several tiles, ragged tails
# ---------------------------------------------------------------------------
SMALL = [
    ("tiny_fp32_full", wl.WORKLOADS["tiny_fp32"], None, (32, 16, 64)),
    ("gqa_shape", wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=1337, pool_blocks=None), None,
     (512, 64, 1024)),
    ("mixed_shape", wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=5, max_len=3000), None,
     (512, 128)),
    ("serving_shape", wl.scaled(wl.WORKLOADS["serving_256"], num_seqs=7, max_len=2500), None,
     (512, 96)),
    ("f16_gqa", wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=777, dtype=torch.float16), None,
     (256,)),
    # long enough that V1 (and V2 at P = 1024) share each item across a cluster
    ("f16_gqa_split", wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=3001, dtype=torch.float16),
     None, (1024,)),
    ("f32_d128", wl.scaled(wl.WORKLOADS["serving_256"], num_seqs=3, max_len=700,
                           dtype=torch.float32), None, (64,)),
]


@pytest.mark.parametrize("name,w,_,parts", SMALL, ids=[s[0] for s in SMALL])
@pytest.mark.parametrize("path,portable", PATH_MODES, ids=[f"{p}{'-portable' if q else ''}"
                                                           for p, q in PATH_MODES])
def test_small_parity(name, w, _, parts, path, portable):
    bc = wl.make(w, poison=True, table_pad=1)
    ref = _ref(bc)
    bg = bc.to("cuda")
    tol = TOL[w.dtype]
    for P in (parts if path == "v2" else parts[:1]):
        got = run(bg, path=path, partition_size=P, portable=portable)
        assert_close(got, ref, tol, f"{name} {path} P={P} portable={portable}")


# Batch sizes that make the reduce take each of its slice widths (32, 64,
# 128 and 256 output elements per CTA for head_dim 256 on a 152-SM GPU; the
# width widens as the batch's rows grow) with 16-token partitions, so that
# rows have up to ~40 partitions and every thread folds several batches.
REDUCE_SHAPES = [(1, 600), (16, 600), (32, 600), (128, 600)]


@pytest.mark.parametrize("num_seqs,max_len", REDUCE_SHAPES,
                         ids=[f"B{b}" for b, _ in REDUCE_SHAPES])
def test_reduce_slice_widths(num_seqs, max_len):
    w = wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=num_seqs, max_len=max_len)
    bc = wl.make(w, poison=True)
    ref = _ref(bc)
    bg = bc.to("cuda")
    for P in (16, 512):
        got = run(bg, path="v2", partition_size=P)
        assert_close(got, ref, TOL[w.dtype], f"B={num_seqs} P={P}")
        # the reduce kernel itself (pa_decode_v2 folds it into pass 1 here)
        got2, _ = _partitions_then_reduce(bg, P, False)
        assert_close(got2, ref, TOL[w.dtype], f"B={num_seqs} P={P} two calls")
        # a bf16 output: the float32 result's bound plus half an ulp of the rounding
        got16 = run(bg, path="v2", partition_size=P, out_dtype=torch.bfloat16)
        assert np.all(np.abs(got16 - ref) <= 2e-3 + np.abs(bf16_round(ref)) * 2.0 ** -8)


@pytest.mark.parametrize("split_x", [False, True], ids=["standard", "split_x"])
@pytest.mark.parametrize("num_seqs", [1024, 1025])
def test_compact_work_list_boundary(num_seqs, split_x):
    """V2 batches of up to 1024 sequences walk a compact list of the
    partitions that exist; larger ones walk the dense (sequence, KV head,
    partition) space.  Both sides of the boundary, and V1 on the same batch,
    against the oracle on every row, on both tensor-core kernels (standard
    and split-x cache layouts)."""
    w = dataclasses.replace(
        wl.WORKLOADS["mixed_32"], name=f"boundary_{num_seqs}", num_seqs=num_seqs, num_heads=8,
        num_kv_heads=2, head_dim=128, block_size=16, pool_blocks=None,
        seq_lens=lambda g, n=num_seqs: torch.randint(1, 601, (n,), generator=g,
                                                     dtype=torch.int64).to(torch.int32))
    bc = wl.make(w, poison=True)
    ref = _ref(bc)
    bg = bc.to("cuda")
    for path, P in (("v2", 256), ("v2", 64), ("v1", 256)):
        assert_close(run(bg, path=path, partition_size=P, split_x=split_x), ref, TOL[w.dtype],
                     f"B={num_seqs} {path} P={P} split_x={split_x}")


def test_v1_v2_agree():
    bc = wl.make(wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=5000), poison=True)
    bg = bc.to("cuda")
    o1 = run(bg, path="v1")
    for P in (64, 512, 1024):
        o2 = run(bg, path="v2", partition_size=P)
        assert max_err(o1, o2) <= 2e-3


def test_dispatch_boundary():
    """max_seq_len 8192 runs V1 and 8193 runs V2 (threshold of the pages),
    both matching the oracle."""
    for L in (8192, 8193):
        w = wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=1, seq_len=L)
        bc = wl.make(w, poison=True)
        params = pa.make_params(bc.q, bc.k_cache, bc.block_tables, max_seq_len=L,
                                scale=bc.scale)
        assert pa.decode_path(params) == (1 if L == 8192 else 2)
        got = run(bc.to("cuda"), path="decode")
        assert_close(got, _ref(bc), 2e-3, f"dispatch L={L}")


def _partitions_then_reduce(bg, P, portable):
    """pa_decode_v2_partitions then pa_decode_v2_reduce on a NaN-poisoned
    workspace: returns (out, workspace)."""
    params = pa.make_params(bg.q, bg.k_cache, bg.block_tables, max_seq_len=bg.max_seq_len,
                            scale=bg.scale, partition_size=P, portable=portable,
                            out_dtype=torch.float32)
    ws = torch.empty(pa.workspace_size(params), dtype=torch.uint8, device="cuda")
    ws.view(torch.float32).fill_(float("nan"))
    pa.workspace_init(ws)
    pa.decode_v2_partitions(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, ws,
                            max_seq_len=bg.max_seq_len, scale=bg.scale, partition_size=P,
                            out_dtype=torch.float32, portable=portable)
    out = torch.full(tuple(bg.q.shape), float("nan"), dtype=torch.float32, device="cuda")
    pa.decode_v2_reduce(params, bg.seq_lens, ws, out)
    torch.cuda.synchronize()
    assert pa.read_device_status(ws, clear=False) == pa.PA_OK
    return out.double().cpu().numpy(), ws


def test_workspace_intermediates_match_partitioned_oracle():
    """Pass 1 alone (pa_decode_v2_partitions): max_logits, exp_sums and
    tmp_output of every partition that exists, against the oracle's Phase 1
    in double; then pass 2 alone (pa_decode_v2_reduce) against the oracle."""
    bc = wl.make(wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=4, max_len=2200), poison=True)
    P = 256
    _, ml_r, es_r, to_r = oracle.decode_partitioned(bc.q, bc.k_cache, bc.v_cache,
                                                    bc.block_tables, bc.seq_lens, bc.scale, P,
                                                    max_partitions=-(-bc.max_seq_len // P))
    ref = _ref(bc)
    for portable in (False, True):
        out, ws = _partitions_then_reduce(bc.to("cuda"), P, portable)
        ml, es, to = workspace_views(ws, bc, P)
        live = np.isfinite(ml_r)
        assert np.all(np.isfinite(ml[live])) and np.all(np.isfinite(to[live]))
        assert max_err(ml[live], ml_r[live]) <= 1e-4 * max(1.0, np.abs(ml_r[live]).max())
        rel = np.abs(es[live] - es_r[live]) / es_r[live]
        assert rel.max() <= 1e-4
        assert max_err(to[live], to_r[live]) <= 2e-3
        assert_close(out, ref, 2e-3, f"partitions + reduce portable={portable}")


def test_single_partition_sequences_finish_in_pass1():
    """Per-sequence V1 / V2 choice inside pa_decode_v2: a sequence of at most
    partition_size tokens is written straight into out by pass 1 (its
    workspace slots stay untouched), longer ones go through the partials and
    the reduce; every row matches the oracle."""
    P = 512
    lens = [1, 100, 512, 513, 2000, 300, 1024, 7]
    w = dataclasses.replace(wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=len(lens)),
                            seq_lens=lambda g: torch.tensor(lens, dtype=torch.int32))
    bc = wl.make(w, poison=True)
    ref = _ref(bc)
    bg = bc.to("cuda")
    for portable in (False, True):
        got, ws = run(bg, path="v2", partition_size=P, portable=portable, return_ws=True)
        assert_close(got, ref, 2e-3, f"per-sequence choice portable={portable}")
        ml, es, to = workspace_views(ws, bc, P)
        for b, L in enumerate(lens):
            if L <= P:   # finished in pass 1: no partials written
                assert np.all(np.isnan(ml[b])) and np.all(np.isnan(to[b])), (b, L)
            else:        # split: every partition's partials written
                n = -(-L // P)
                assert np.all(np.isfinite(ml[b, :, :n])) and np.all(np.isfinite(to[b, :, :n]))
        # the two-call form writes the partials of every sequence and agrees
        got2, ws2 = _partitions_then_reduce(bg, P, portable)
        assert_close(got2, ref, 2e-3, f"partitions + reduce portable={portable}")
        assert max_err(got, got2) <= 2e-3
        ml2, _, _ = workspace_views(ws2, bc, P)
        assert all(np.all(np.isfinite(ml2[b, :, :-(-L // P)])) for b, L in enumerate(lens))


def test_block_permutation_is_bit_identical():
    bc = wl.make(wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=3001), poison=False)
    nb = bc.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(5))
    k2 = torch.empty_like(bc.k_cache)
    v2 = torch.empty_like(bc.v_cache)
    k2[perm] = bc.k_cache
    v2[perm] = bc.v_cache
    bt2 = perm[bc.block_tables.long()].to(torch.int32)
    b1 = bc.to("cuda")
    b2 = wl.Batch(bc.workload, bc.q, k2, v2, bt2, bc.seq_lens, bc.max_seq_len).to("cuda")
    for path, portable in PATH_MODES:
        o1 = run(b1, path=path, portable=portable)
        o2 = run(b2, path=path, portable=portable)
        assert np.array_equal(o1, o2), f"{path} portable={portable}"


def test_repeat_runs_are_bit_identical():
    bg = wl.make(wl.scaled(wl.WORKLOADS["serving_256"], num_seqs=9, max_len=4000)).to("cuda")
    for path, portable in PATH_MODES:
        first = run(bg, path=path, portable=portable)
        for _ in range(3):
            assert np.array_equal(run(bg, path=path, portable=portable), first)


def test_concurrent_host_threads():
    """Calls are thread-safe: four host threads, each with its own stream,
    workspace and batch, decode concurrently (ctypes releases the GIL during
    the calls); every result is bit-identical to the same batch decoded alone
    and matches the oracle."""
    import threading
    batches = [wl.make(wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=3, max_len=L))
               for L in (900, 3000, 9000, 20000)]
    refs = [_ref(b) for b in batches]
    alone = [run(b.to("cuda"), path="decode") for b in batches]
    results, errors = {}, []

    def worker(i):
        try:
            bg = batches[i].to("cuda")
            stream = torch.cuda.Stream()
            params = pa.make_params(bg.q, bg.k_cache, bg.block_tables, max_seq_len=bg.max_seq_len,
                                    scale=bg.scale, out_dtype=torch.float32)
            ws = pa.alloc_workspace(params, device="cuda")
            out = torch.empty(tuple(bg.q.shape), dtype=torch.float32, device="cuda")
            torch.cuda.synchronize()
            with torch.cuda.stream(stream):
                for _ in range(20):
                    pa.decode(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws,
                              max_seq_len=bg.max_seq_len, scale=bg.scale, stream=stream)
            stream.synchronize()
            assert pa.read_device_status(ws) == pa.PA_OK
            results[i] = out.double().cpu().numpy()
        except Exception as e:  # reported below, in the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(batches))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for i in range(len(batches)):
        assert np.array_equal(results[i], alone[i])
        assert_close(results[i], refs[i], 2e-3, f"thread {i}")


@pytest.mark.parametrize("split_x", [False, True], ids=["standard", "split_x"])
def test_bf16_output(split_x):
    """A bf16 `out` on every way the tensor-core kernels write it: V1 (in
    clusters for one 2100-token sequence), V2 through the reduce kernel, and
    the one-launch V2 step (a 30000-token sequence), on both cache
    layouts."""
    cases = [(wl.scaled(wl.WORKLOADS["gqa_8k"], seq_len=2100), ("v1", "v2")),
             (wl.scaled(wl.WORKLOADS["long_100k"], seq_len=30000), ("v2",))]
    for w, paths in cases:
        bc = wl.make(w, poison=True)
        ref = _ref(bc)
        bg = bc.to("cuda")
        for path in paths:
            got = run(bg, path=path, out_dtype=torch.bfloat16, split_x=split_x)
            # float32 result within 2e-3, then one bf16 rounding: half an ulp more
            ulp_half = np.abs(bf16_round(ref)) * 2.0 ** -8
            assert np.all(np.abs(got - ref) <= 2e-3 + ulp_half), (w.name, path, split_x)


# ---------------------------------------------------------------------------
# edge cases
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("path,portable", PATH_MODES)
def test_edge_lengths(path, portable):
    """L = 1, a block boundary, a partition boundary, a partition plus one,
    and a zero-length sequence (zero row) in one batch."""
    lens = (1, 16, 512, 513, 0, 1023, 31)
    bc = problem(dtype=torch.bfloat16, lens=lens, Hq=24, Hkv=4, D=256, BS=16, seed=7)
    ref = _ref(bc)
    got = run(bc.to("cuda"), path=path, partition_size=512, portable=portable)
    assert np.all(got[4] == 0.0)
    assert_close(got, ref, 2e-3, f"edge lengths {path}")


def test_single_key_gives_value_row():
    bc = problem(dtype=torch.bfloat16, lens=(1, 1, 1), Hq=6, Hkv=1, D=128, BS=32, seed=8)
    for path, portable in PATH_MODES:
        got = run(bc.to("cuda"), path=path, portable=portable)
        for s in range(3):
            v0 = bc.v_cache[int(bc.block_tables[s, 0]), 0, 0].double().numpy()
            for h in range(6):
                assert np.array_equal(got[s, h], v0), (path, portable)


def test_partition_larger_than_sequence():
    bc = problem(dtype=torch.bfloat16, lens=(300, 77), Hq=8, Hkv=2, D=64, BS=16, seed=9)
    ref = _ref(bc)
    got = run(bc.to("cuda"), path="v2", partition_size=4096)
    assert_close(got, ref, 2e-3, "P > L")


def test_empty_batch():
    bc = problem(dtype=torch.bfloat16, lens=(), Hq=8, Hkv=2, D=64, BS=16, seed=10, pool=4)
    bg = bc.to("cuda")
    out = torch.empty((0, 8, 64), dtype=torch.float32, device="cuda")
    pa.decode(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, None,
              max_seq_len=0, scale=bc.scale)
    torch.cuda.synchronize()


def test_large_logits_stay_finite():
    w = wl.scaled(wl.WORKLOADS["long_100k"], seq_len=20000)
    bc = wl.make(dataclasses_replace(w, key_outlier_frac=0.002), poison=True)
    ref = _ref(bc)
    for path, portable in PATH_MODES:
        got = run(bc.to("cuda"), path=path, portable=portable)
        assert_close(got, ref, 2e-3, f"outliers {path} portable={portable}")


def dataclasses_replace(w, **kw):
    import dataclasses
    return dataclasses.replace(w, **kw)


def test_bad_block_id_poisons_the_row_and_sets_status():
    bc = problem(dtype=torch.bfloat16, lens=(100, 100), Hq=4, Hkv=2, D=64, BS=16, seed=11)
    bc.block_tables[1, 2] = bc.k_cache.shape[0] + 5          # outside the pool
    ref = _ref(problem(dtype=torch.bfloat16, lens=(100, 100), Hq=4, Hkv=2, D=64, BS=16, seed=11))
    bg = bc.to("cuda")
    for path, portable in PATH_MODES:
        got, ws = run(bg, path="v2" if path == "v2" else "v1", portable=portable,
                      partition_size=32, return_ws=True, check_status=False)
        assert np.all(np.isnan(got[1])), path
        assert_close(got[0], ref[0], 2e-3, "untouched row")
        if path == "v2":
            assert pa.read_device_status(ws) == pa.PA_ERR_BAD_BLOCK_ID
            assert pa.read_device_status(ws) == pa.PA_OK      # cleared by the read


def test_bad_seq_len_poisons_the_row_and_sets_status():
    bc = problem(dtype=torch.bfloat16, lens=(60, 60), Hq=4, Hkv=2, D=64, BS=16, seed=12)
    bg = bc.to("cuda")
    bg.seq_lens[1] = 61                                       # > max_seq_len promised
    ref = _ref(bc)
    for path, portable in PATH_MODES:
        got, ws = run(bg, path=path, portable=portable, partition_size=32, return_ws=True,
                      check_status=False)
        assert np.all(np.isnan(got[1])), path
        assert_close(got[0], ref[0], 2e-3, "untouched row")
        if path == "v2":
            assert pa.read_device_status(ws) == pa.PA_ERR_BAD_SEQ_LEN


def test_bad_inputs_on_split_items():
    """Tensor-core shapes whose items are shared by a cluster of CTAs (V1 and
    small V2 batches): a bad block id inside one CTA's share poisons the
    whole row, a bad seq_len poisons its row, the other rows stay exact."""
    lens = (3000, 2500, 2000)
    good = problem(dtype=torch.bfloat16, lens=lens, Hq=12, Hkv=2, D=256, BS=16, seed=13)
    ref = _ref(good)
    bc = problem(dtype=torch.bfloat16, lens=lens, Hq=12, Hkv=2, D=256, BS=16, seed=13)
    bc.block_tables[0, 150] = -7                              # token 2400: a late share
    bg = bc.to("cuda")
    bg.seq_lens[2] = 3001                                     # > max_seq_len promised
    for path in ("v1", "v2"):
        got, ws = run(bg, path=path, partition_size=1024, return_ws=True, check_status=False)
        assert np.all(np.isnan(got[0])), path
        assert np.all(np.isnan(got[2])), path
        assert_close(got[1], ref[1], 2e-3, f"untouched row {path}")
        if path == "v2":
            assert pa.read_device_status(ws) in (pa.PA_ERR_BAD_BLOCK_ID, pa.PA_ERR_BAD_SEQ_LEN)


# ---------------------------------------------------------------------------
# the five workloads at full size, in the launch configuration bench.py times
# ---------------------------------------------------------------------------
FULL = ["tiny_fp32", "gqa_8k", "long_100k", "mixed_32", "serving_256"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    """Every row of the workload at full size against the oracle, through
    pa_decode (the bench's launch) and V2 where pa_decode picks V1; and V1
    forced on the long batches, which must match both the oracle and V2
    within the same bound (its clusters split a 100K-token sequence)."""
    w = wl.WORKLOADS[name]
    bg = wl.make(w, device="cuda", poison=True)
    bc = bg.to("cpu")
    tol = TOL[w.dtype]
    ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens, bc.scale)
    v1_default = bg.max_seq_len <= pa.DEFAULT_V1_MAX_SEQ_LEN
    for P in w.partition_sizes:
        for path in ("decode", "v2") if v1_default else ("decode",):
            got = run(bg, path=path, partition_size=P)
            assert_close(got, ref, tol, f"{name} {path} P={P}")
    if not v1_default:
        o1 = run(bg, path="v1")
        assert_close(o1, ref, tol, f"{name} v1")
        o2 = run(bg, path="v2", partition_size=w.partition_sizes[0])
        assert max_err(o1, o2) <= tol, f"{name}: V1 and V2 differ by {max_err(o1, o2):.3e}"


def test_decode_from_host_buffers_matches_device_call():
    """pa_decode_host (host q / block table / lengths / out, pinned) gives the
    same bits as pa_decode on device copies of the same inputs, on both
    paths."""
    for L, v1max in ((3000, pa.DEFAULT_V1_MAX_SEQ_LEN), (3000, 1024)):
        bc = wl.make(wl.scaled(wl.WORKLOADS["mixed_32"], num_seqs=3, max_len=L), poison=True)
        bg = bc.to("cuda")
        params = pa.make_params(bc.q, bc.k_cache, bc.block_tables, max_seq_len=bc.max_seq_len,
                                scale=bc.scale, out_dtype=torch.float32, v1_max_seq_len=v1max)
        ws = pa.alloc_workspace(params) if pa.decode_path(params) == 2 else None
        ref = run(bg, path="decode", v1_max_seq_len=v1max)
        staging = pa.alloc_host_staging(params)
        out_h = torch.empty(tuple(bc.q.shape), dtype=torch.float32).pin_memory()
        pa.decode_host(bc.q.pin_memory(), bg.k_cache, bg.v_cache, bc.block_tables.pin_memory(),
                       bc.seq_lens.pin_memory(), out_h, ws, staging, max_seq_len=bc.max_seq_len,
                       scale=bc.scale, v1_max_seq_len=v1max)
        assert np.array_equal(out_h.double().numpy(), ref), f"path {pa.decode_path(params)}"
        # the inputs in a pinned mirror of the staging layout (one copy in)
        _, qm, btm, slm = pa.alloc_host_mirror(params, bc.q.dtype, *bc.q.shape,
                                               bc.block_tables.shape[1])
        qm.copy_(bc.q)
        btm.copy_(bc.block_tables)
        slm.copy_(bc.seq_lens)
        out_h.fill_(float("nan"))
        pa.decode_host(qm, bg.k_cache, bg.v_cache, btm, slm, out_h, ws, staging,
                       max_seq_len=bc.max_seq_len, scale=bc.scale, v1_max_seq_len=v1max)
        assert np.array_equal(out_h.double().numpy(), ref), "mirrored host inputs"
        if ws is not None:
            assert pa.read_device_status(ws) == pa.PA_OK


def test_cuda_graph_capture_and_replay():
    """pa_decode captured once in a CUDA graph (V2 with its programmatic-
    dependent reduce, and V1 with clustered CTAs) and replayed with new q and
    shorter sequence lengths copied into the captured buffers: every replay
    matches the oracle on that replay's inputs."""
    cases = [(wl.scaled(wl.WORKLOADS["long_100k"], seq_len=20000), 512),
             (wl.WORKLOADS["gqa_8k"], 512)]
    for w, P in cases:
        bc = wl.make(w, poison=True)
        bg = bc.to("cuda")
        params = pa.make_params(bc.q, bc.k_cache, bc.block_tables, max_seq_len=bc.max_seq_len,
                                scale=bc.scale, partition_size=P, out_dtype=torch.float32)
        ws = pa.alloc_workspace(params) if pa.decode_path(params) == 2 else None
        out = torch.empty(tuple(bc.q.shape), device="cuda")
        kw = dict(max_seq_len=bc.max_seq_len, scale=bc.scale, partition_size=P)
        pa.decode(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws, **kw)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            pa.decode(bg.q, bg.k_cache, bg.v_cache, bg.block_tables, bg.seq_lens, out, ws, **kw)
        g = torch.Generator().manual_seed(77)
        for cut in (0, 777, 4099):
            q_new = torch.randn(tuple(bc.q.shape), generator=g).to(bc.q.dtype)
            lens = (bc.seq_lens - cut).clamp(min=1)
            bg.q.copy_(q_new)
            bg.seq_lens.copy_(lens)
            graph.replay()
            torch.cuda.synchronize()
            ref = oracle.decode(q_new, bc.k_cache, bc.v_cache, bc.block_tables, lens, bc.scale)
            assert_close(out.double().cpu().numpy(), ref, 2e-3,
                         f"graph replay path {pa.decode_path(params)} cut {cut}")
        if ws is not None:
            assert pa.read_device_status(ws) == pa.PA_OK


@pytest.mark.parametrize("dtype,D,BS", [(torch.bfloat16, 256, 16), (torch.float16, 128, 32),
                                        (torch.bfloat16, 64, 32), (torch.float32, 64, 16),
                                        (torch.float32, 256, 32), (torch.bfloat16, 64, 8)])
def test_split_x_layout(dtype, D, BS):
    """PA_FLAG_SPLIT_X: the caches in the pages' V1 layout, read directly, on
    V1, V2 and pa_decode.  The CUDA-core kernels (PA_FLAG_PORTABLE, and the
    only kernels for float32 or block size 8) give the same bits as on the
    standard layout; the split-x tensor-core kernel (bf16 / f16, block 16 or
    32) matches the oracle and the CUDA-core kernels within the tolerance."""
    lens = (1, BS - 1, 300, 777, 0, 1500)
    bc = problem(dtype=dtype, lens=lens, Hq=12, Hkv=3, D=D, BS=BS, seed=21)
    ref = _ref(bc)
    bg = bc.to("cuda")
    k5, v4 = (t.cuda() for t in split_x_caches(bc))
    kw = dict(max_seq_len=bc.max_seq_len, scale=bc.scale)
    tensor_core = dtype != torch.float32 and BS in (16, 32)
    params = pa.make_params(bc.q, k5, bc.block_tables, partition_size=256,
                            out_dtype=torch.float32, split_x=True, **kw)
    assert pa.decode_kernel(params) == (2 if tensor_core else 1)
    for path in ("v1", "v2", "decode"):
        want = run(bg, path=path, partition_size=256, portable=True, v1_max_seq_len=1024)
        for portable in ((False, True) if tensor_core else (True,)):
            got = torch.full(tuple(bc.q.shape), float("nan"), device="cuda")
            ws = pa.alloc_workspace(params)
            kx = dict(split_x=True, portable=portable, **kw)
            if path == "v1":
                pa.decode_v1(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, **kx)
            elif path == "v2":
                pa.decode_v2(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, ws,
                             partition_size=256, **kx)
            else:
                pa.decode(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, ws, partition_size=256,
                          v1_max_seq_len=1024, **kx)
            torch.cuda.synchronize()
            g = got.double().cpu().numpy()
            what = f"split-x {path} {'CUDA-core' if portable else 'tensor-core'}"
            if portable:
                assert np.array_equal(g, want), f"{what} differs from the standard layout"
            else:
                assert max_err(g, want) <= TOL[dtype], what
            assert_close(g, ref, TOL[dtype], what)
            assert pa.read_device_status(ws) == pa.PA_OK


@pytest.mark.parametrize("dtype,D,BS", [(torch.bfloat16, 128, 16), (torch.float16, 64, 32)])
def test_split_x_persistent_walk(dtype, D, BS):
    """More split-x work items than two per SM, so each CTA of the persistent
    grid walks several items (its ring streams from one item into the next,
    its two q tiles alternate): V1 and V2 on every row against the oracle,
    and a block id outside the pool, planted in one sequence, poisons that
    sequence's rows only (the CTAs that meet it go on to correct items)."""
    gen = torch.Generator().manual_seed(5)
    lens = torch.randint(0, 2000, (96,), generator=gen).tolist()
    lens[:11] = [0, 1, BS - 1, BS, BS + 1, 256, 257, 1999, 1024, 700, 1500]
    bad_seq = 10
    kw = dict(dtype=dtype, lens=lens, Hq=16, Hkv=4, D=D, BS=BS, seed=31)
    ref = _ref(problem(**kw))
    bc = problem(**kw)
    bc.block_tables[bad_seq, 3] = bc.k_cache.shape[0] + 1     # outside the pool
    bg = bc.to("cuda")
    k5, v4 = (t.cuda() for t in split_x_caches(bc))
    kx = dict(max_seq_len=bc.max_seq_len, scale=bc.scale, split_x=True)
    params = pa.make_params(bc.q, k5, bc.block_tables, partition_size=256,
                            out_dtype=torch.float32, **kx)
    assert pa.decode_kernel(params) == 2
    keep = [b for b in range(len(lens)) if b != bad_seq]
    for path in ("v1", "v2"):
        got = torch.full(tuple(bc.q.shape), float("nan"), device="cuda")
        ws = pa.alloc_workspace(params)
        if path == "v1":
            pa.decode_v1(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, **kx)
        else:
            pa.decode_v2(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, ws,
                         partition_size=256, **kx)
        torch.cuda.synchronize()
        g = got.double().cpu().numpy()
        assert np.all(np.isnan(g[bad_seq])), path
        assert_close(g[keep], ref[keep], TOL[dtype], f"split-x persistent {path}")
        if path == "v2":
            assert pa.read_device_status(ws) == pa.PA_ERR_BAD_BLOCK_ID


def test_split_x_clusters_share_items():
    """Fewer split-x work items than SMs: a cluster of CTAs shares each item
    and merges the shares through distributed shared memory.  V1 (clusters
    of 8 here) on lengths that leave some CTAs of a cluster without tokens
    (5 and 0 tokens), V2 at P = 4096 (clusters of 4, then the reduce), and
    the one-sequence 8192-token workload through pa_decode (V1, clusters of
    16): every row against the oracle, and a block id outside the pool in
    one CTA's share poisons only its sequence."""
    lens = (8192, 5, 0, 3001)
    kw = dict(dtype=torch.bfloat16, lens=lens, Hq=24, Hkv=4, D=256, BS=16, seed=41)
    ref = _ref(problem(**kw))
    bc = problem(**kw)
    bad_seq = 3
    bc.block_tables[bad_seq, 100] = bc.k_cache.shape[0] + 3   # token 1600: a middle share
    bg = bc.to("cuda")
    k5, v4 = (t.cuda() for t in split_x_caches(bc))
    kx = dict(max_seq_len=bc.max_seq_len, scale=bc.scale, split_x=True)
    keep = [b for b in range(len(lens)) if b != bad_seq]
    got = torch.full(tuple(bc.q.shape), float("nan"), device="cuda")
    pa.decode_v1(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, **kx)
    torch.cuda.synchronize()
    g = got.double().cpu().numpy()
    assert np.all(np.isnan(g[bad_seq]))
    assert_close(g[keep], ref[keep], TOL[torch.bfloat16], "split-x V1 in clusters")
    assert np.all(g[2] == 0.0)                                  # the empty sequence
    params = pa.make_params(bc.q, k5, bc.block_tables, partition_size=4096,
                            out_dtype=torch.float32, **kx)
    ws = pa.alloc_workspace(params)
    got.fill_(float("nan"))
    pa.decode_v2(bg.q, k5, v4, bg.block_tables, bg.seq_lens, got, ws, partition_size=4096, **kx)
    torch.cuda.synchronize()
    g = got.double().cpu().numpy()
    assert np.all(np.isnan(g[bad_seq]))
    assert_close(g[keep], ref[keep], TOL[torch.bfloat16], "split-x V2 in clusters")
    assert pa.read_device_status(ws) == pa.PA_ERR_BAD_BLOCK_ID
    # config 2's shape: one 8192-token sequence, pa_decode -> V1
    w = wl.WORKLOADS["gqa_8k"]
    bc2 = wl.make(w, poison=True)
    bg2 = bc2.to("cuda")
    k5, v4 = split_x_caches(bg2)
    params = pa.make_params(bg2.q, k5, bg2.block_tables, max_seq_len=bg2.max_seq_len,
                            scale=bg2.scale, out_dtype=torch.float32, split_x=True)
    assert pa.decode_path(params) == 1 and pa.decode_kernel(params) == 2
    got = torch.full(tuple(bg2.q.shape), float("nan"), device="cuda")
    pa.decode(bg2.q, k5, v4, bg2.block_tables, bg2.seq_lens, got, None,   # V1: no workspace
              max_seq_len=bg2.max_seq_len, scale=bg2.scale, split_x=True)
    torch.cuda.synchronize()
    assert_close(got.double().cpu().numpy(), _ref(bc2), TOL[w.dtype], "split-x gqa_8k V1")


def test_split_x_full_size_long_context():
    """The 100K-token long-context workload with its caches rewritten (on the
    device, as test input) into the split-x layout: pa_decode (V2) on the
    split-x tensor-core kernel against the oracle on every row, in the launch
    configuration the bench times (784 items on the persistent grid)."""
    w = wl.WORKLOADS["long_100k"]
    bg = wl.make(w, device="cuda", poison=True)
    bc = bg.to("cpu")
    ref = oracle.decode(bc.q, bc.k_cache, bc.v_cache, bc.block_tables, bc.seq_lens, bc.scale)
    k5, v4 = split_x_caches(bg)
    params = pa.make_params(bg.q, k5, bg.block_tables, max_seq_len=bg.max_seq_len,
                            scale=bg.scale, partition_size=512, out_dtype=torch.float32,
                            split_x=True)
    assert pa.decode_kernel(params) == 2 and pa.decode_path(params) == 2
    ws = pa.alloc_workspace(params)
    out = torch.full(tuple(bg.q.shape), float("nan"), device="cuda")
    pa.decode(bg.q, k5, v4, bg.block_tables, bg.seq_lens, out, ws, max_seq_len=bg.max_seq_len,
              scale=bg.scale, partition_size=512, split_x=True)
    torch.cuda.synchronize()
    assert_close(out.double().cpu().numpy(), ref, TOL[w.dtype], "split-x long_100k")
    assert pa.read_device_status(ws) == pa.PA_OK


# ---------------------------------------------------------------------------
# V2 in one launch: the pass-1 grid runs pass 2 itself after its streaming
# ---------------------------------------------------------------------------
def _one_launch_cases():
    lens = [20000, 1, 0, 512, 513, 9000]
    mixed = dataclasses.replace(
        wl.WORKLOADS["mixed_32"], name="mixed_small_heads", num_seqs=len(lens), num_heads=8,
        num_kv_heads=2, head_dim=128, block_size=16, pool_blocks=None,
        seq_lens=lambda g: torch.tensor(lens, dtype=torch.int32))
    return [(wl.scaled(wl.WORKLOADS["long_100k"], seq_len=30000), 512),   # 59 partitions
            (mixed, 128),                       # lengths 0 .. 20000: direct, zero and split rows
            (wl.scaled(wl.WORKLOADS["long_100k"], seq_len=60000), 1024)]  # two rounds of items


@pytest.mark.parametrize("split_x", [False, True], ids=["standard", "split_x"])
@pytest.mark.parametrize("case", [0, 1, 2], ids=["one_long_sequence", "mixed_lengths",
                                                 "two_rounds"])
def test_one_launch_back_to_back_then_graph_replay(case, split_x):
    """pa_decode_v2 as one launch, on the standard and on the split-x cache
    layout (each its own tensor-core kernel): two steps in a row on one
    NaN-poisoned workspace with different q and lengths, then the step
    captured in a CUDA graph and replayed twice with new inputs; every step
    against the oracle, and after each launch the control block ready for
    the next (marker intact, epoch advanced by one, start count back at
    zero)."""
    w, P = _one_launch_cases()[case]
    bc = wl.make(w, poison=True)
    bg = bc.to("cuda")
    kc, vc = split_x_caches(bg) if split_x else (bg.k_cache, bg.v_cache)
    params = pa.make_params(bc.q, kc, bc.block_tables, max_seq_len=bc.max_seq_len,
                            scale=bc.scale, partition_size=P, out_dtype=torch.float32,
                            v1_max_seq_len=1, split_x=split_x)    # pa_decode's choice: V2
    assert pa.decode_launches(params) == 1 and pa.decode_kernel(params) == 2
    ws = torch.empty(pa.workspace_size(params), dtype=torch.uint8, device="cuda")
    ws.view(torch.float32).fill_(float("nan"))
    pa.workspace_init(ws)
    out = torch.full(tuple(bc.q.shape), float("nan"), device="cuda")
    kw = dict(max_seq_len=bc.max_seq_len, scale=bc.scale, partition_size=P, split_x=split_x)
    g = torch.Generator().manual_seed(90 + case)
    launches = [0]

    def new_inputs(cut):
        q = torch.randn(tuple(bc.q.shape), generator=g).to(bc.q.dtype)
        lens = torch.where(bc.seq_lens > cut, bc.seq_lens - cut, bc.seq_lens)
        bg.q.copy_(q)
        bg.seq_lens.copy_(lens)
        return q, lens

    def check(q, lens, what):
        launches[0] += 1
        ref = oracle.decode(q, bc.k_cache, bc.v_cache, bc.block_tables, lens, bc.scale)
        assert_close(out.double().cpu().numpy(), ref, TOL[w.dtype], what)
        assert pa.read_device_status(ws, clear=False) == pa.PA_OK
        marker, epoch, started, _, _ = control_words(ws)
        assert (marker, epoch, started) == (MARKER, launches[0], 0), (what, epoch, started)

    for step, cut in enumerate((0, 333)):
        q, lens = new_inputs(cut)
        pa.decode_v2(bg.q, kc, vc, bg.block_tables, bg.seq_lens, out, ws, **kw)
        torch.cuda.synchronize()
        check(q, lens, f"step {step}")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        pa.decode_v2(bg.q, kc, vc, bg.block_tables, bg.seq_lens, out, ws, **kw)
    for rep, cut in enumerate((1000, 7)):
        q, lens = new_inputs(cut)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        check(q, lens, f"replay {rep}")


def test_one_launch_matches_two_launches_closely():
    """The one-launch step and the two-kernel form (pa_decode_v2_partitions,
    pa_decode_v2_reduce) compute the same log-sum-exp identity in different
    orders: they agree far inside the tolerance, and each is bit-identical
    from run to run."""
    bg = wl.make(wl.scaled(wl.WORKLOADS["long_100k"], seq_len=50000), poison=True).to("cuda")
    params = pa.make_params(bg.q, bg.k_cache, bg.block_tables, max_seq_len=bg.max_seq_len,
                            scale=bg.scale, partition_size=256, out_dtype=torch.float32)
    assert pa.decode_launches(params) == 1
    one = run(bg, path="v2", partition_size=256)           # 196 partitions
    two, _ = _partitions_then_reduce(bg, 256, False)
    assert max_err(one, two) <= 1e-5
    assert np.array_equal(run(bg, path="v2", partition_size=256), one)


@pytest.mark.parametrize("split_x", [False, True], ids=["standard", "split_x"])
def test_uninitialised_workspace_is_reported_not_reduced(split_x):
    """A workspace that pa_workspace_init never initialised (NaN everywhere,
    control block included): the one-launch step reduces nothing, the status
    word reads PA_ERR_WORKSPACE_NOT_INIT, the rows it would have reduced
    (split sequences, and the empty one) are NaN, and the sequence that pass
    1 finished itself is still right (both cache layouts)."""
    lens = [3000, 100, 0, 5000]
    w = dataclasses.replace(
        wl.WORKLOADS["mixed_32"], name="uninit", num_seqs=len(lens), num_heads=8,
        num_kv_heads=2, head_dim=128, block_size=16, pool_blocks=None,
        seq_lens=lambda g: torch.tensor(lens, dtype=torch.int32))
    bc = wl.make(w, poison=True)
    ref = _ref(bc)
    bg = bc.to("cuda")
    params = pa.make_params(bc.q, split_x_caches(bc)[0] if split_x else bc.k_cache,
                            bc.block_tables, max_seq_len=bc.max_seq_len, scale=bc.scale,
                            partition_size=128, out_dtype=torch.float32, v1_max_seq_len=1,
                            split_x=split_x)                      # pa_decode's choice: V2
    assert pa.decode_launches(params) == 1
    ws = torch.empty(pa.workspace_size(params), dtype=torch.uint8, device="cuda")
    ws.view(torch.float32).fill_(float("nan"))
    got = run(bg, path="v2", partition_size=128, workspace=ws, check_status=False,
              split_x=split_x)
    assert pa.read_device_status(ws) == pa.PA_ERR_WORKSPACE_NOT_INIT
    for b, L in enumerate(lens):
        if L > 128 or L == 0:
            assert np.all(np.isnan(got[b])), b
        else:
            assert_close(got[b], ref[b], 2e-3, f"sequence {b} (L={L})")
    # once initialised, the same workspace gives the right answer
    pa.workspace_init(ws)
    assert_close(run(bg, path="v2", partition_size=128, workspace=ws, split_x=split_x), ref,
                 2e-3, "after init")


def test_two_launches_for_many_rows():
    """A batch with more reduce units (query rows x head_dim / 32) than the
    persistent grid has CTAs -- 2048 sequences x 8 heads -- runs as pass 1
    plus the dependent reduce kernel; every row against the oracle."""
    n = 2048
    w = dataclasses.replace(
        wl.WORKLOADS["mixed_32"], name="many_heads", num_seqs=n, num_heads=8, num_kv_heads=8,
        head_dim=128, block_size=16, pool_blocks=None,
        seq_lens=lambda g: torch.randint(1, 301, (n,), generator=g,
                                         dtype=torch.int64).to(torch.int32))
    bc = wl.make(w, poison=True)
    params = pa.make_params(bc.q, bc.k_cache, bc.block_tables, max_seq_len=bc.max_seq_len,
                            scale=bc.scale, partition_size=16, out_dtype=torch.float32,
                            v1_max_seq_len=1)                     # pa_decode's choice: V2
    assert pa.decode_launches(params) == 2
    assert_close(run(bc.to("cuda"), path="v2", partition_size=16), _ref(bc), 2e-3, "two launches")
