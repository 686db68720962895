"""Host-side checks of the benchmark's bookkeeping (CPU only): the
algorithmic bytes and FLOPs it divides by, against hand counts, and the
reference arm's JSON line."""
import dataclasses
import json
import os
import subprocess
import sys

import pytest
import torch

from paged_attention_decode_v2_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def test_decode_algorithmic_bytes_hand_count():
    """Every K and V element of each sequence once, plus q: with 24 query /
    4 KV heads, head_dim 256 and 2-byte elements a token costs
    4 * 256 * 2 (K and V) * 2 bytes = 4096 B."""
    w = wl.scaled(wl.WORKLOADS["gqa_8k"], num_seqs=3)
    w = dataclasses.replace(w, seq_lens=lambda g: torch.tensor([1, 100, 1000], dtype=torch.int32))
    b = wl.make(w)
    assert b.kv_bytes() == (1 + 100 + 1000) * 4096
    assert b.q_bytes() == 3 * 24 * 256 * 2
    # the 100K workload's figure quoted with the results
    assert 100000 * 4096 + 24 * 256 * 2 == 409_612_288


def test_prefill_flops_hand_count():
    """Query i of a chunk sees its C cached tokens and chunk tokens 0..i:
    contexts (3, 0) with chunks (2, 3) give (3+1) + (3+2) + 1 + 2 + 3 = 15
    visible (query, key) pairs per head, each costing 4 * head_dim FLOPs."""
    pw = wl.prefill_problem(dtype=torch.bfloat16, ctx=(3, 0), new=(2, 3), Hq=6, Hkv=2, D=128)
    pb = wl.make_prefill(pw)
    assert bench.prefill_flops(pb) == 4 * 128 * 6 * 15
    w = wl.PREFILL_WORKLOADS["prefill_32k"]
    n, C = 8192, 24576
    assert 4 * 256 * 24 * (n * C + n * (n + 1) // 2) == 5_772_536_709_120
    assert w.num_heads == 24 and w.head_dim == 256


def test_traffic_lookup_is_keyed_to_sources():
    """A recorded DRAM figure is reported only for the sources it was taken
    on: any other hash, workload or path gives None."""
    for (kernel, h, workload, P, path), v in bench.NCU_TRAFFIC.items():
        assert kernel in bench.KERNEL_SOURCES and v > 0
        assert bench.ncu_traffic(kernel, workload, P, "no-such-path") is None
    assert bench.ncu_traffic("pa_tc_kernel", "long_100k", 4096, "v2") is None
    assert bench.ncu_traffic("no_such_kernel", "long_100k", 512, "v2") is None


@pytest.mark.timeout(300)
def test_reference_arm_prints_one_json_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny_fp32", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["unit"] == bench.UNIT
    assert d["metric"] == bench.METRIC and d["higher_is_better"] is False
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_traffic_key_ignores_comments_not_code():
    """The ncu traffic table is keyed by the kernels' code with comments and
    layout left out: editing a comment or re-wrapping a line keeps the key,
    a change of code (or of a string literal, as in inline assembly) does
    not, and comment markers inside a string literal are code."""
    src = 'int f(int x) {  // doubles x\n  /* the\n  body */ return 2 * x;\n}\nconst char* s = "a // b";\n'
    same = 'int f(int x) {\n    /* twice x */\n  return 2 *   x; }  // end\nconst char* s = "a // b";\n'
    code = src.replace("2 * x", "3 * x")
    lit = src.replace('"a // b"', '"a // c"')
    k = bench._code_only
    assert k(src) == k(same)
    assert k(src) != k(code)
    assert k(src) != k(lit)
    assert "// b" in k(src) and "doubles" not in k(src) and "body" not in k(src)
    # every listed kernel hashes, and the table's keys name listed kernels
    for name in bench.KERNEL_SOURCES:
        assert len(bench.kernel_source_hash(name)) == 16
    assert all(key[0] in bench.KERNEL_SOURCES for key in bench.NCU_TRAFFIC)
