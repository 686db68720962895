"""Pins of the float64 oracle to facts that do not come from the oracle itself.

Each ``pin_*`` function takes an :class:`oracle.Oracle` and raises
``AssertionError`` if the oracle disagrees with what the pages or plain
mathematics fix.  ``test_oracle_pins.py`` runs them on the real oracle;
``test_oracle_mutants.py`` runs them on copies with planted mistakes and
requires that every mistake trips at least one pin.

The pages describe the computation in commit 4eb83a7e "qwen3_6_scripts",
paragraph "Implementation (paged_attention_v2_pytorch.py)" (Phase 1: per
partition QK^T, softmax, weighted V; Phase 2: global max, rescale by
exp(m_p - global_max) * exp_sum_p, weighted sum) and check V1 against plain
("manual") attention in the paragraph "V1 paged_attention (decode <= 8192)".
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

from paged_attention_decode_v2_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def problem(dtype=torch.float32, lens=(37,), Hq=6, Hkv=2, D=16, BS=4, seed=0, pool=None,
            poison=True, table_pad=1, outlier_frac=0.0, outlier_scale=1.0):
    """A small seeded paged batch (NaN-poisoned outside its tokens by default)."""
    lens = tuple(int(x) for x in lens)
    w = wl.Workload("pin", dtype, len(lens), Hq, Hkv, D, BS, (BS,), seed,
                    lambda g, l=lens: torch.tensor(l, dtype=torch.int32), pool_blocks=pool,
                    key_outlier_frac=outlier_frac, key_outlier_scale=outlier_scale)
    return wl.make(w, poison=poison, table_pad=table_pad)


def dense_reference(batch, scale=None):
    """Brute force: gather each sequence's keys/values to dense [L, D] with
    torch indexing and call the library's scaled_dot_product_attention in
    float64 (an implementation the oracle does not share)."""
    w = batch.workload
    scale = batch.scale if scale is None else scale
    G = w.num_heads // w.num_kv_heads
    out = torch.zeros(w.num_seqs, w.num_heads, w.head_dim, dtype=torch.float64)
    for b in range(w.num_seqs):
        L = int(batch.seq_lens[b])
        if L == 0:
            continue
        t = torch.arange(L)
        blk = batch.block_tables[b, t // w.block_size].long()
        off = t % w.block_size
        for h in range(w.num_heads):
            kvh = h // G
            K = batch.k_cache[blk, kvh, off].double()
            V = batch.v_cache[blk, kvh, off].double()
            qh = batch.q[b, h].double()
            o = F.scaled_dot_product_attention(qh[None, None, None, :], K[None, None],
                                               V[None, None], scale=scale)
            out[b, h] = o[0, 0, 0]
    return out.numpy()


def _run(orc, batch, scale=None):
    s = batch.scale if scale is None else scale
    return orc.decode(batch.q, batch.k_cache, batch.v_cache, batch.block_tables,
                      batch.seq_lens, s)


def _close(a, b, tol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    assert np.all(np.isfinite(a)), f"{what}: non-finite values"
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"


# --------------------------------------------------------------------------
# (P5) brute force on tiny inputs, every dtype, GQA groups, ragged tails
# --------------------------------------------------------------------------
def pin_brute_force(orc):
    cases = [
        dict(dtype=torch.float32, lens=(37,), Hq=6, Hkv=2, D=16, BS=4, seed=1),
        dict(dtype=torch.bfloat16, lens=(1, 5, 16, 33), Hq=4, Hkv=2, D=8, BS=8, seed=2),
        dict(dtype=torch.float16, lens=(23, 9), Hq=3, Hkv=1, D=12, BS=4, seed=3),
        dict(dtype=torch.float32, lens=(50,), Hq=8, Hkv=4, D=32, BS=16, seed=4),
    ]
    for c in cases:
        b = problem(**c)
        _close(_run(orc, b), dense_reference(b), 1e-12, f"brute force {c}")
    # a scale that is not 1/sqrt(D)
    b = problem(dtype=torch.float32, lens=(19,), Hq=2, Hkv=1, D=8, BS=4, seed=5)
    _close(_run(orc, b, scale=0.73), dense_reference(b, scale=0.73), 1e-12, "brute force scale")


# --------------------------------------------------------------------------
# (P1) partitioned (Phase 1 + Phase 2) equals unpartitioned attention
# --------------------------------------------------------------------------
def pin_partition_identity(orc):
    for dtype, lens, BS in ((torch.float32, (100,), 16), (torch.bfloat16, (1, 31, 64, 65), 8)):
        b = problem(dtype=dtype, lens=lens, Hq=4, Hkv=2, D=16, BS=BS, seed=11)
        ref = _run(orc, b)
        for P in (BS, 2 * BS, 3 * BS, 32, 48, 512, 10**6):
            out, ml, es, to = orc.decode_partitioned(b.q, b.k_cache, b.v_cache, b.block_tables,
                                                     b.seq_lens, b.scale, P)
            _close(out, ref, 1e-12, f"partition identity P={P} {dtype}")
            # workspace shape: exactly ceil(L/P) partitions per sequence are written
            for i, L in enumerate(lens):
                n = -(-L // P)
                assert np.all(np.isfinite(ml[i, :, :n])), "missing partition"
                assert np.all(np.isnan(ml[i, :, n:])), "partition past the sequence written"
                # every partition's exp-sum is in [1, tokens in partition]
                cnt = np.minimum(P, L - P * np.arange(n))
                assert np.all(es[i, :, :n] >= 1.0 - 1e-12)
                assert np.all(es[i, :, :n] <= cnt[None, :] + 1e-9)


# --------------------------------------------------------------------------
# (P2) one key: the output is that token's value row, exactly
# --------------------------------------------------------------------------
def pin_single_key(orc):
    for dtype in (torch.float32, torch.bfloat16, torch.float16):
        b = problem(dtype=dtype, lens=(1, 1), Hq=4, Hkv=2, D=8, BS=4, seed=21)
        out = _run(orc, b)
        for s in range(2):
            blk = int(b.block_tables[s, 0])
            for h in range(4):
                v0 = b.v_cache[blk, h // 2, 0].double().numpy()
                assert np.array_equal(out[s, h], v0), f"single key {dtype}"
        out_p = orc.decode_partitioned(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                       b.scale, 4)[0]
        assert np.array_equal(out_p, out), "single key partitioned"


# --------------------------------------------------------------------------
# (P3) identical keys, or scale 0: the output is the mean of the value rows
# --------------------------------------------------------------------------
def _value_mean(b):
    w = b.workload
    G = w.num_heads // w.num_kv_heads
    out = np.zeros((w.num_seqs, w.num_heads, w.head_dim))
    for s in range(w.num_seqs):
        L = int(b.seq_lens[s])
        rows = [b.v_cache[int(b.block_tables[s, t // w.block_size]), :, t % w.block_size]
                .double().numpy() for t in range(L)]
        m = np.mean(np.stack(rows), axis=0)  # [Hkv, D]
        for h in range(w.num_heads):
            out[s, h] = m[h // G]
    return out


def pin_identical_keys(orc):
    b = problem(dtype=torch.float32, lens=(29, 7), Hq=4, Hkv=2, D=8, BS=4, seed=31)
    w = b.workload
    # make every key of every sequence equal to one vector per KV head
    for s in range(w.num_seqs):
        L = int(b.seq_lens[s])
        for t in range(L):
            blk = int(b.block_tables[s, t // w.block_size])
            b.k_cache[blk, :, t % w.block_size] = torch.arange(w.head_dim) * 0.25 - 1.0
    _close(_run(orc, b), _value_mean(b), 1e-13, "identical keys")
    b2 = problem(dtype=torch.bfloat16, lens=(40, 3), Hq=6, Hkv=3, D=8, BS=8, seed=32)
    _close(_run(orc, b2, scale=0.0), _value_mean(b2), 1e-13, "scale 0")
    out_p = orc.decode_partitioned(b2.q, b2.k_cache, b2.v_cache, b2.block_tables, b2.seq_lens,
                                   0.0, 16)[0]
    _close(out_p, _value_mean(b2), 1e-13, "scale 0 partitioned")


# --------------------------------------------------------------------------
# (P4) physical block placement does not change the result, bit for bit
# --------------------------------------------------------------------------
def pin_block_permutation(orc):
    b = problem(dtype=torch.bfloat16, lens=(45, 12, 64), Hq=4, Hkv=2, D=16, BS=8, seed=41,
                poison=False, table_pad=0)
    ref = _run(orc, b)
    ref_p = orc.decode_partitioned(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                   b.scale, 16)[0]
    nb = b.k_cache.shape[0]
    g = torch.Generator().manual_seed(42)
    perm = torch.randperm(nb, generator=g)          # new position of old block i
    k2 = torch.empty_like(b.k_cache)
    v2 = torch.empty_like(b.v_cache)
    k2[perm] = b.k_cache
    v2[perm] = b.v_cache
    bt2 = perm[b.block_tables.long()].to(torch.int32)
    out = orc.decode(b.q, k2, v2, bt2, b.seq_lens, b.scale)
    assert np.array_equal(out, ref), "block permutation changed the direct result"
    out_p = orc.decode_partitioned(b.q, k2, v2, bt2, b.seq_lens, b.scale, 16)[0]
    assert np.array_equal(out_p, ref_p), "block permutation changed the partitioned result"


# --------------------------------------------------------------------------
# (P6) adding one vector u to every key shifts each head's logits by a
#      constant, which softmax ignores
# --------------------------------------------------------------------------
def pin_shift_invariance(orc):
    b = problem(dtype=torch.float32, lens=(33, 17), Hq=4, Hkv=2, D=8, BS=4, seed=61)
    g = torch.Generator().manual_seed(62)
    # put q, k on a dyadic grid so that k + u is exact in float32
    b.q.copy_(torch.randint(-8, 9, b.q.shape, generator=g).float() / 8)
    b.k_cache.copy_(torch.nan_to_num(b.k_cache).clamp(-4, 4).mul(8).round().div(8))
    ref = _run(orc, b, scale=0.5)
    u = torch.randint(-4, 5, (b.k_cache.shape[1], 1, b.k_cache.shape[3]), generator=g).float()
    k2 = b.k_cache + u / 4
    out = orc.decode(b.q, k2, b.v_cache, b.block_tables, b.seq_lens, 0.5)
    _close(out, ref, 1e-12, "shift invariance")
    out_p = orc.decode_partitioned(b.q, k2, b.v_cache, b.block_tables, b.seq_lens, 0.5, 8)[0]
    _close(out_p, ref, 1e-12, "shift invariance partitioned")


# --------------------------------------------------------------------------
# (P7) large logits: max subtraction keeps the result finite; one dominant
#      key gives that key's value row
# --------------------------------------------------------------------------
def pin_large_logits(orc):
    b = problem(dtype=torch.float32, lens=(70,), Hq=2, Hkv=1, D=8, BS=8, seed=71)
    w = b.workload
    t_star = 52                                   # lies in partition 3 of 16-token partitions
    blk = int(b.block_tables[0, t_star // w.block_size])
    b.q[0].fill_(1.0)
    b.k_cache[blk, 0, t_star % w.block_size] = 400.0   # logit = 400 * 8 * scale
    out = _run(orc, b, scale=1.0)
    v_star = b.v_cache[blk, 0, t_star % w.block_size].double().numpy()
    for h in range(2):
        _close(out[0, h], v_star, 1e-12, "dominant key")
    out_p = orc.decode_partitioned(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                   1.0, 16)[0]
    for h in range(2):
        _close(out_p[0, h], v_star, 1e-12, "dominant key partitioned")
    # 0.1% (here: a few) of keys scaled by 30, as in the long-context batch
    b2 = problem(dtype=torch.bfloat16, lens=(3000,), Hq=2, Hkv=1, D=16, BS=16, seed=72,
                 outlier_frac=0.002, outlier_scale=30.0)
    out2 = _run(orc, b2)
    _close(out2, dense_reference(b2), 1e-12, "outlier keys")
    out2p = orc.decode_partitioned(b2.q, b2.k_cache, b2.v_cache, b2.block_tables, b2.seq_lens,
                                   b2.scale, 512)[0]
    _close(out2p, out2, 1e-12, "outlier keys partitioned")


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------
def pin_closed_forms(orc):
    # three keys whose logits are 0, 1, 2: weights 1 : e : e^2
    D, BS = 4, 2
    k = torch.zeros(4, 1, BS, D)
    v = torch.zeros(4, 1, BS, D)
    table = torch.tensor([[3, 1]], dtype=torch.int32)   # tokens 0,1 in block 3; token 2 in 1
    k[3, 0, 0] = torch.tensor([0.0, 0.0, 0.0, 0.0])
    k[3, 0, 1] = torch.tensor([1.0, 0.0, 0.0, 0.0])
    k[1, 0, 0] = torch.tensor([2.0, 0.0, 0.0, 0.0])
    vals = [[1.0, -2.0, 0.5, 3.0], [4.0, 0.0, -1.0, 2.0], [-3.0, 1.0, 2.0, 0.25]]
    v[3, 0, 0] = torch.tensor(vals[0])
    v[3, 0, 1] = torch.tensor(vals[1])
    v[1, 0, 0] = torch.tensor(vals[2])
    q = torch.tensor([[[1.0, 5.0, -7.0, 9.0]]])
    lens = torch.tensor([3], dtype=torch.int32)
    e = math.e
    want = [(vals[0][d] + e * vals[1][d] + e * e * vals[2][d]) / (1 + e + e * e) for d in range(D)]
    out = orc.decode(q, k, v, table, lens, 1.0)
    _close(out[0, 0], want, 1e-14, "three-key closed form")
    for P in (2, 4):
        outp = orc.decode_partitioned(q, k, v, table, lens, 1.0, P)[0]
        _close(outp[0, 0], want, 1e-14, f"three-key closed form P={P}")
    # two keys: the output is v0 + sigmoid(l1 - l0) (v1 - v0)
    lens2 = torch.tensor([2], dtype=torch.int32)
    out2 = orc.decode(q, k, v, table, lens2, 0.5)
    sig = 1.0 / (1.0 + math.exp(-0.5))
    want2 = [vals[0][d] + sig * (vals[1][d] - vals[0][d]) for d in range(D)]
    _close(out2[0, 0], want2, 1e-14, "two-key closed form")


# --------------------------------------------------------------------------
# degenerate cases: empty batch, zero-length sequence, bad block ids
# --------------------------------------------------------------------------
def pin_degenerate(orc):
    b = problem(dtype=torch.float32, lens=(9, 0, 4), Hq=2, Hkv=1, D=8, BS=4, seed=81)
    out = _run(orc, b)
    assert np.all(out[1] == 0.0), "zero-length sequence must give a zero row"
    _close(out[[0, 2]], dense_reference(b)[[0, 2]], 1e-12, "rows beside an empty sequence")
    empty = problem(dtype=torch.float32, lens=(), Hq=2, Hkv=1, D=8, BS=4, seed=82, pool=4)
    assert _run(orc, empty).shape == (0, 2, 8)
    bad = problem(dtype=torch.float32, lens=(9,), Hq=2, Hkv=1, D=8, BS=4, seed=83)
    bad.block_tables[0, 1] = bad.k_cache.shape[0]          # one past the pool
    try:
        _run(orc, bad)
    except ValueError:
        pass
    else:
        raise AssertionError("a block id outside the pool must be rejected")


# --------------------------------------------------------------------------
# the pages' printed partition counts (tests/golden/partition_counts.json)
# --------------------------------------------------------------------------
def pin_golden_partition_counts(orc):
    with open(os.path.join(GOLDEN, "partition_counts.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        L, P = c["seq_len"], c["partition_size"]
        b = problem(dtype=torch.bfloat16, lens=(L,), Hq=1, Hkv=1, D=8, BS=16, seed=91,
                    poison=False, table_pad=0)
        _, ml, _, _ = orc.decode_partitioned(b.q, b.k_cache, b.v_cache, b.block_tables,
                                             b.seq_lens, b.scale, P,
                                             max_partitions=c["num_partitions"] + 4)
        written = int(np.isfinite(ml[0, 0]).sum())
        assert written == c["num_partitions"], f"L={L} P={P}: {written} partitions"
        last = L - (written - 1) * P
        assert last == c["last_partition_tokens"], f"last partition has {last} tokens"


# --------------------------------------------------------------------------
# paged prefix prefill (commit 1a4e1005 "paged_attn.py", opening paragraph;
# commit 4eb83a7e "qwen3_6_scripts", paragraphs on the prefix attention's
# pre-allocated buffers, "Complete rewrite ..." item 1, "Prefill
# (flash_attn_func)": context from the paged cache, the chunk causal)
# --------------------------------------------------------------------------
def _prefill(orc, pb, **kw):
    return orc.prefill(pb.q, pb.k, pb.v, pb.k_cache, pb.v_cache, pb.block_tables,
                       pb.query_start, pb.ctx_lens, pb.scale, **kw)


def _prefill_dense(pb):
    """Brute force with torch: gather each sequence's context from the cache
    by indexing, append the chunk's keys / values, and call
    scaled_dot_product_attention in float64 with an explicit boolean mask
    (context visible, chunk lower-triangular)."""
    w = pb.workload
    G = w.num_heads // w.num_kv_heads
    T = pb.q.shape[0]
    out = torch.zeros(T, w.num_heads, w.head_dim, dtype=torch.float64)
    for b in range(w.num_seqs):
        C = int(pb.ctx_lens[b])
        s0, s1 = int(pb.query_start[b]), int(pb.query_start[b + 1])
        n = s1 - s0
        if n == 0:
            continue
        t = torch.arange(C)
        blk = pb.block_tables[b, t // w.block_size].long()
        off = t % w.block_size
        for h in range(w.num_heads):
            kvh = h // G
            K = torch.cat([pb.k_cache[blk, kvh, off].double(), pb.k[s0:s1, kvh].double()])
            V = torch.cat([pb.v_cache[blk, kvh, off].double(), pb.v[s0:s1, kvh].double()])
            Q = pb.q[s0:s1, h].double()
            mask = torch.ones(n, C + n, dtype=torch.bool)
            mask[:, C:] = torch.tril(torch.ones(n, n, dtype=torch.bool))
            o = F.scaled_dot_product_attention(Q[None, None], K[None, None], V[None, None],
                                               attn_mask=mask[None, None], scale=pb.scale)
            out[s0:s1, h] = o[0, 0]
    return out.numpy()


def pin_prefill_brute_force(orc):
    """Against torch SDPA with an explicit mask, for batches mixing an empty
    context, ragged contexts and chunks, GQA and each element type."""
    for dtype, ctx, new, Hq, Hkv, D, BS in (
            (torch.float32, (23, 0, 40), (9, 13, 1), 6, 2, 16, 4),
            (torch.bfloat16, (50, 7), (20, 33), 4, 4, 32, 16),
            (torch.float16, (0,), (29,), 3, 1, 8, 8)):
        pb = wl.make_prefill(wl.prefill_problem(dtype=dtype, ctx=ctx, new=new, Hq=Hq, Hkv=Hkv,
                                                D=D, BS=BS, seed=41), poison=True)
        _close(_prefill(orc, pb), _prefill_dense(pb), 1e-12, f"prefill brute force {dtype}")


def pin_prefill_one_token_is_decode(orc):
    """A chunk of one token after C cached ones is a single-token decode over
    C + 1 tokens: write the token's key / value into slot C of a decode
    cache and compare with the decode oracle (itself pinned above)."""
    lens = (41, 1, 16)
    d = problem(dtype=torch.float32, lens=lens, Hq=6, Hkv=3, D=16, BS=4, seed=17, poison=False)
    B = len(lens)
    pos = torch.tensor([L - 1 for L in lens])
    blk = d.block_tables[torch.arange(B), pos // 4].long()
    off = pos % 4
    k_new = d.k_cache[blk, :, off].clone()          # [B, Hkv, D]: the last token's rows
    v_new = d.v_cache[blk, :, off].clone()
    kc, vc = d.k_cache.clone(), d.v_cache.clone()
    kc[blk, :, off] = float("nan")                   # the prefill must not read slot C
    vc[blk, :, off] = float("nan")
    pw = wl.prefill_problem(dtype=torch.float32, ctx=[L - 1 for L in lens], new=[1] * B,
                            Hq=6, Hkv=3, D=16, BS=4)
    pb = wl.PrefillBatch(pw, d.q.clone(), k_new, v_new, kc, vc, d.block_tables,
                         torch.arange(B + 1, dtype=torch.int32),
                         torch.tensor([L - 1 for L in lens], dtype=torch.int32), 1, max(lens) - 1)
    _close(_prefill(orc, pb), _run(orc, d), 1e-12, "one-token prefill vs decode")


def pin_prefill_no_context_is_causal(orc):
    """With no cached context the chunk is plain causal self-attention:
    torch SDPA with is_causal=True (GQA by repeating each KV head over its
    query heads)."""
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.float32, ctx=(0, 0), new=(31, 12),
                                            Hq=6, Hkv=2, D=16, BS=4, seed=5))
    got = _prefill(orc, pb)
    G = 3
    for b in range(2):
        s0, s1 = int(pb.query_start[b]), int(pb.query_start[b + 1])
        Q = pb.q[s0:s1].double().transpose(0, 1)                        # [Hq, n, D]
        K = pb.k[s0:s1].double().transpose(0, 1).repeat_interleave(G, 0)
        V = pb.v[s0:s1].double().transpose(0, 1).repeat_interleave(G, 0)
        ref = F.scaled_dot_product_attention(Q, K, V, is_causal=True, scale=pb.scale)
        _close(got[s0:s1], ref.transpose(0, 1).numpy(), 1e-12, f"causal sequence {b}")


def pin_prefill_prefix_means(orc):
    """Closed form: with q = 0 every visible logit is 0, so row i is the
    plain mean of the context values and of the chunk values 0..i."""
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.float32, ctx=(10, 0), new=(6, 4),
                                            Hq=2, Hkv=1, D=4, BS=4, seed=8))
    pb.q.zero_()
    got = _prefill(orc, pb)
    for b in range(2):
        C = int(pb.ctx_lens[b])
        s0, s1 = int(pb.query_start[b]), int(pb.query_start[b + 1])
        t = torch.arange(C)
        ctx_v = pb.v_cache[pb.block_tables[b, t // 4].long(), 0, t % 4].double()
        for i in range(s1 - s0):
            vis = torch.cat([ctx_v, pb.v[s0:s0 + i + 1, 0].double()])
            for h in range(2):
                _close(got[s0 + i, h], vis.mean(0).numpy(), 1e-13, f"prefix mean b={b} i={i}")


def pin_prefill_causality(orc):
    """Changing the key and value of chunk token j changes the rows of tokens
    i >= j of that sequence only."""
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.float32, ctx=(9, 5), new=(8, 6),
                                            Hq=2, Hkv=1, D=8, BS=4, seed=12))
    base = _prefill(orc, pb)
    j = int(pb.query_start[0]) + 4
    pb.k[j] += 3.0
    pb.v[j] -= 2.0
    moved = np.abs(_prefill(orc, pb) - base).max(axis=(1, 2)) > 0
    expect = np.zeros(pb.q.shape[0], dtype=bool)
    expect[j:int(pb.query_start[1])] = True
    assert np.array_equal(moved, expect), f"rows changed: {np.nonzero(moved)[0].tolist()}"


def pin_prefill_tiled_is_direct(orc):
    """The pages' tiled online softmax (context tiles, then chunk tiles,
    with m_blk / m_new / corr) reaches the plain definition for any tile."""
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.bfloat16, ctx=(45, 0, 16), new=(20, 9, 3),
                                            Hq=4, Hkv=2, D=16, BS=8, seed=23), poison=True)
    direct = _prefill(orc, pb)
    for tile in (1, 7, 16, 128):
        tiled = orc.prefill_tiled(pb.q, pb.k, pb.v, pb.k_cache, pb.v_cache, pb.block_tables,
                                  pb.query_start, pb.ctx_lens, pb.scale, tile)
        _close(tiled, direct, 1e-13, f"tiled prefill, tile {tile}")


# --------------------------------------------------------------------------
# the subset mode (rows=) the full-size tests and the CPU baseline use
# --------------------------------------------------------------------------
def pin_rows_subset(orc):
    """Asking for a list of rows (any order, repeats allowed) gives exactly
    those rows of the full output, bit for bit: the subset mode computes the
    same rows, not different ones, and puts row r of the request at r."""
    b = problem(dtype=torch.bfloat16, lens=(37, 1, 64, 20), Hq=6, Hkv=2, D=16, BS=8, seed=61)
    full = _run(orc, b).reshape(-1, 16)
    rows = [23, 0, 5, 5, 17, 6, 12, 1, 22]
    sub = orc.decode(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.scale, rows=rows)
    assert sub.shape == (len(rows), 16), sub.shape
    assert np.array_equal(sub, full[rows]), "decode rows= differs from the full output's rows"
    pb = wl.make_prefill(wl.prefill_problem(dtype=torch.float16, ctx=(19, 0), new=(7, 5), Hq=4,
                                            Hkv=2, D=8, BS=4, seed=62), poison=True)
    fullp = _prefill(orc, pb).reshape(-1, 8)
    rows = [47, 3, 3, 0, 28, 30, 11]
    subp = _prefill(orc, pb, rows=rows)
    assert subp.shape == (len(rows), 8), subp.shape
    assert np.array_equal(subp, fullp[rows]), "prefill rows= differs from the full output's rows"


ALL_PINS = [
    pin_rows_subset,
    pin_prefill_brute_force,
    pin_prefill_one_token_is_decode,
    pin_prefill_no_context_is_causal,
    pin_prefill_prefix_means,
    pin_prefill_causality,
    pin_prefill_tiled_is_direct,
    pin_brute_force,
    pin_partition_identity,
    pin_single_key,
    pin_identical_keys,
    pin_block_permutation,
    pin_shift_invariance,
    pin_large_logits,
    pin_closed_forms,
    pin_degenerate,
    pin_golden_partition_counts,
]
