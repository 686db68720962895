"""GPU parity of the paged prefix prefill (pa_prefill) against the float64 oracle.

Tolerance, derived from the kernel's arithmetic: logits are exact products
summed in float32, so their error is negligible next to the one rounding of
p = 2^(s - m) to the 16-bit element type before P.V.  The kernel divides by
the sum of the *rounded* p, so its output is an exact weighted mean of the
visible values with every weight perturbed by a relative error of at most u
(2^-8 for bf16, 2^-11 for f16).  Such a mean moves by at most
2u / (1 - u) * max_j |v_j - o| per element, where o is the exact output and j
runs over the row's visible keys; the test checks every element against that
bound (plus 2e-5 for the float32 accumulation) and also that the typical
error stays far below it.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import paged_attention_decode_v2_gb300 as pa
from paged_attention_decode_v2_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

UNIT_ROUNDOFF = {torch.bfloat16: 2.0 ** -8, torch.float16: 2.0 ** -11}


@pytest.fixture(scope="module", autouse=True)
def _built():
    from paged_attention_decode_v2_gb300 import build
    build.build()
    assert torch.cuda.is_available(), "the gpu tests need a CUDA device"


def _ref(pb, rows=None):
    return oracle.prefill(pb.q, pb.k, pb.v, pb.k_cache, pb.v_cache, pb.block_tables,
                          pb.query_start, pb.ctx_lens, pb.scale, rows=rows)


def _run(pb, out_dtype=torch.float32, fill=float("nan"), **kw):
    g = pb.to("cuda")
    out = torch.full(tuple(g.q.shape), fill, dtype=out_dtype, device="cuda")
    args = dict(max_query_len=pb.max_query_len, max_ctx_len=pb.max_ctx_len, scale=pb.scale)
    args.update(kw)
    pa.prefill(g.q, g.k, g.v, g.k_cache, g.v_cache, g.block_tables, g.query_start, g.ctx_lens,
               out, **args)
    torch.cuda.synchronize()
    return out.double().cpu().numpy()


def _bound(pb, ref):
    """Per-element bound 2u/(1-u) * max_j |v_j - o| over each row's visible
    values (cumulative max / min of the context + chunk values)."""
    w = pb.workload
    u = UNIT_ROUNDOFF[w.dtype]
    G = w.num_heads // w.num_kv_heads
    spread = np.zeros_like(ref)
    for b in range(w.num_seqs):
        C = int(pb.ctx_lens[b])
        s0, s1 = int(pb.query_start[b]), int(pb.query_start[b + 1])
        if s1 == s0:
            continue
        t = torch.arange(C)
        blk = pb.block_tables[b, t // w.block_size].long()
        off = t % w.block_size
        for kvh in range(w.num_kv_heads):
            vals = torch.cat([pb.v_cache[blk, kvh, off].double(), pb.v[s0:s1, kvh].double()])
            hi = torch.cummax(vals, 0).values[C:].numpy()   # row i: max over keys < C + i + 1
            lo = torch.cummin(vals, 0).values[C:].numpy()
            for h in range(kvh * G, (kvh + 1) * G):
                o = ref[s0:s1, h]
                spread[s0:s1, h] = np.maximum(hi - o, o - lo)
    return 2 * u / (1 - u) * spread + 2e-5


def _check(pb, got, ref, what):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    bound = _bound(pb, ref)
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"{what}: error {worst:.3f} x the rounding bound"
    # the bound is a worst case; random data sits far below it
    assert float(np.mean(err)) <= 0.05 * float(np.mean(bound)), f"{what}: mean error too large"
    return float(np.max(err))


# (name, dtype, ctx lens, chunk lens, Hq, Hkv, D, BS)
CASES = [
    ("bf16_d256_gqa6", torch.bfloat16, (0, 300, 1000), (200, 129, 37), 24, 4, 256, 16),
    ("f16_d128_mha", torch.float16, (130, 0), (256, 300), 8, 8, 128, 32),
    ("bf16_d128_g8_bs64", torch.bfloat16, (64, 777), (1, 129), 16, 2, 128, 64),
    ("bf16_d256_bs32_long_ctx", torch.bfloat16, (4096,), (513,), 4, 1, 256, 32),
    ("f16_d256_ragged", torch.float16, (17, 2047, 5), (127, 128, 385), 6, 2, 256, 16),
]


@pytest.mark.parametrize("name,dtype,ctx,new,Hq,Hkv,D,BS", CASES, ids=[c[0] for c in CASES])
def test_prefill_parity(name, dtype, ctx, new, Hq, Hkv, D, BS):
    pb = wl.make_prefill(wl.prefill_problem(dtype=dtype, ctx=ctx, new=new, Hq=Hq, Hkv=Hkv, D=D,
                                            BS=BS, seed=len(name)), poison=True)
    ref = _ref(pb)
    got = _run(pb)
    _check(pb, got, ref, name)
    # the same call again gives the same bits
    assert np.array_equal(_run(pb), got)


def test_prefill_16bit_output():
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=(333,), new=(150,), Hq=6,
                                            Hkv=2, D=128, BS=16, seed=3), poison=True)
    ref = _ref(pb)
    got = _run(pb, out_dtype=torch.bfloat16)
    # plus one rounding of the output to bf16
    bound = _bound(pb, ref) + np.abs(ref) * 2.0 ** -8
    assert np.all(np.abs(got - ref) <= bound)


def test_prefill_block_permutation_is_bit_identical():
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=(700, 90), new=(140, 60),
                                            Hq=8, Hkv=2, D=128, BS=16, seed=9))
    nb = pb.k_cache.shape[0]
    perm = torch.randperm(nb, generator=torch.Generator().manual_seed(4))
    k2 = torch.empty_like(pb.k_cache)
    v2 = torch.empty_like(pb.v_cache)
    k2[perm] = pb.k_cache
    v2[perm] = pb.v_cache
    pb2 = dataclasses.replace(pb, k_cache=k2, v_cache=v2,
                              block_tables=perm[pb.block_tables.long()].to(torch.int32))
    assert np.array_equal(_run(pb), _run(pb2))


def test_prefill_bad_inputs():
    """A context block id outside the pool or a context length past
    max_ctx_len makes that sequence's rows NaN; a chunk longer than
    max_query_len leaves its rows untouched; the other sequences are exact."""
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=(300, 200, 100, 50),
                                            new=(40, 30, 20, 10), Hq=4, Hkv=2, D=128, BS=16,
                                            seed=21))
    ref = _ref(pb)
    bt = pb.block_tables.clone()
    bt[0, 5] = -3                                   # context token 80 of sequence 0
    cl = pb.ctx_lens.clone()
    cl[1] = pb.max_ctx_len + 1                      # past the promised bound
    qs = pb.query_start.clone()
    bad = dataclasses.replace(pb, block_tables=bt, ctx_lens=cl)
    got = _run(bad, fill=7.0)
    s = [int(x) for x in qs]
    assert np.all(np.isnan(got[s[0]:s[1]])) and np.all(np.isnan(got[s[1]:s[2]]))
    assert np.max(np.abs(got[s[2]:] - ref[s[2]:])) <= 4e-3
    # chunk of sequence 3 longer than max_query_len: rows left as they were
    got = _run(pb, fill=7.0, max_query_len=9)
    assert np.all(got[s[3]:s[4]] == 7.0)


def test_prefill_unit_orders():
    """Both unit walks of the kernel cover every unit exactly once.  A batch
    with few (cost level, sequence) pairs is walked by cost; 65 sequences
    with contexts near 16K tokens (129+ levels x 65 sequences > 8192 pairs)
    take the query-tile order.  Mixed chunk and context lengths, a 1-token
    chunk and an empty chunk in each."""
    g = torch.Generator().manual_seed(31)
    for nseq, ctx_hi, new_hi in ((6, 3000, 260), (65, 16400, 40)):
        ctx = [int(x) for x in torch.randint(0, ctx_hi, (nseq,), generator=g)]
        new = [int(x) for x in torch.randint(1, new_hi, (nseq,), generator=g)]
        ctx[0], new[0] = ctx_hi, 1
        new[1] = 0
        pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=tuple(ctx),
                                                new=tuple(new), Hq=4, Hkv=2, D=128, BS=16,
                                                seed=nseq), poison=True)
        levels = -(-pb.max_ctx_len // 128) + -(-pb.max_query_len // 128)
        assert (levels * nseq <= 8192) == (nseq == 6)
        _check(pb, _run(pb), _ref(pb), f"{nseq} sequences")


def test_prefill_empty_chunks_and_contexts():
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=(0, 64, 0), new=(0, 5, 1),
                                            Hq=4, Hkv=4, D=128, BS=16, seed=2), poison=True)
    ref = _ref(pb)
    got = _run(pb)
    _check(pb, got, ref, "empty chunks / contexts")


def _bound_rows(pb, rows, ref_rows):
    """The per-element bound of :func:`_bound` for a list of flat rows
    (t * Hq + h) whose oracle outputs are ``ref_rows`` [len(rows), D]."""
    w = pb.workload
    u = UNIT_ROUNDOFF[w.dtype]
    G = w.num_heads // w.num_kv_heads
    qs = [int(x) for x in pb.query_start]
    ext = {}   # (b, kvh) -> running max / min over the sequence's visible values
    out = np.empty_like(ref_rows)
    for r, row in enumerate(rows):
        t, h = divmod(row, w.num_heads)
        b = max(i for i in range(w.num_seqs) if qs[i] <= t)
        kvh = h // G
        if (b, kvh) not in ext:
            C = int(pb.ctx_lens[b])
            tt = torch.arange(C)
            blk = pb.block_tables[b, tt // w.block_size].long()
            vals = torch.cat([pb.v_cache[blk, kvh, tt % w.block_size].double(),
                              pb.v[qs[b]:qs[b + 1], kvh].double()])
            ext[(b, kvh)] = (C, torch.cummax(vals, 0).values.numpy(),
                             torch.cummin(vals, 0).values.numpy())
        C, hi, lo = ext[(b, kvh)]
        i = C + (t - qs[b])          # last visible key of row t
        o = ref_rows[r]
        out[r] = np.maximum(hi[i] - o, o - lo[i])
    return 2 * u / (1 - u) * out + 2e-5


def test_prefill_full_size_tile_edge_rows():
    """prefill_32k (one 8192-token chunk after 24576 cached tokens, 24 / 4
    heads, head_dim 256) in the launch the benchmark times, against the
    oracle on the first and last row of every 128-query tile plus seeded
    random rows, on all 24 heads, each element within the derived rounding
    bound (the same bound as the small cases)."""
    w = wl.PREFILL_WORKLOADS["prefill_32k"]
    pb = wl.make_prefill(w)
    T = pb.q.shape[0]
    g = np.random.default_rng(7)
    toks = sorted({t for q0 in range(0, T, 128) for t in (q0, min(q0 + 127, T - 1))} |
                  set(int(x) for x in g.integers(0, T, 32)))
    rows = [t * w.num_heads + h for t in toks for h in range(w.num_heads)]
    ref = _ref(pb, rows=rows)
    got = _run(pb).reshape(-1, w.head_dim)[rows]
    assert np.all(np.isfinite(got))
    err = np.abs(got - ref)
    bound = _bound_rows(pb, rows, ref)
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"full size: error {worst:.3f} x the rounding bound"
    assert float(np.mean(err)) <= 0.05 * float(np.mean(bound)), "full size: mean error too large"
