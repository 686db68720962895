"""Host side of the C ABI (CPU only: no call here reaches a kernel launch).

Every call below either is a pure host function or fails a host-side check
before anything is enqueued, so these tests run without a GPU.
"""
import ctypes
import json
import os
import re

import pytest

import paged_attention_decode_v2_gb300 as pa
from paged_attention_decode_v2_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "pa.h")
GOLDEN = os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="module")
def L():
    pa_build.build()
    return pa.lib()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"PA_API\s+[\w\s\*]*?\b(pa_\w+)\s*\(", text)))


def test_header_declares_the_abi():
    syms = declared_symbols()
    assert set(syms) == set(pa.EXPORTS), syms


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), f"libpa.so does not export {name}"


def params(**kw):
    base = dict(num_seqs=1, num_heads=24, num_kv_heads=4, head_dim=256, block_size=16,
                num_blocks=6875, max_blocks_per_seq=6250, max_seq_len=100000, partition_size=512,
                v1_max_seq_len=0, kv_dtype=pa.PA_BF16, out_dtype=pa.PA_F32, scale=1 / 16, flags=0)
    base.update(kw)
    return pa.Params(**base)


CONTROL = 1024          # status word, init marker and one-launch counters


def expected_ws(B, H, D, NP):
    r = lambda x: (x + 255) // 256 * 256
    return CONTROL + 2 * r(B * H * NP * 4) + r(B * H * NP * D * 4)


def test_workspace_size_formula(L):
    for P, NP in ((512, 196), (1024, 98)):
        assert pa.workspace_size(params(partition_size=P)) == expected_ws(1, 24, 256, NP)
    p5 = params(num_seqs=256, num_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                num_blocks=40000, max_blocks_per_seq=4096, max_seq_len=131072)
    assert pa.workspace_size(p5) == expected_ws(256, 32, 128, 256)
    # invalid parameters give 0
    assert pa.workspace_size(params(partition_size=500)) == 0      # not a multiple of 16
    assert pa.workspace_size(params(num_kv_heads=5)) == 0          # 24 % 5 != 0


def test_workspace_matches_the_pages_sizing(L):
    g = json.load(open(os.path.join(GOLDEN, "workspace_sizes.json")))
    c, printed = g["case"], g["printed"]
    p = params(num_seqs=c["num_seqs"], num_heads=c["num_heads"], head_dim=c["head_dim"],
               max_seq_len=c["max_seq_len"], partition_size=c["partition_size"],
               max_blocks_per_seq=c["max_seq_len"] // 16, num_blocks=c["max_seq_len"] // 16)
    total = pa.workspace_size(p)
    # regions: control block | max_logits | exp_sums | tmp_output, each 256-aligned
    r = lambda x: (x + 255) // 256 * 256
    assert printed["exp_sums_bytes"] == c["num_seqs"] * c["num_heads"] * c["num_partitions"] * 4
    tmp = total - CONTROL - 2 * r(printed["exp_sums_bytes"])
    assert tmp == 2 * printed["tmp_output_bytes_2B"]          # float32 partials
    assert tmp // 4 == printed["tmp_output_elements"]


def test_dispatch_threshold(L):
    # the pages: seq_len > 8192 -> V2, <= 8192 -> V1
    assert pa.decode_path(params(max_seq_len=8192)) == 1
    assert pa.decode_path(params(max_seq_len=8193)) == 2
    assert pa.decode_path(params(max_seq_len=1)) == 1
    assert pa.decode_path(params(max_seq_len=0)) == 1
    assert pa.decode_path(params(max_seq_len=100000)) == 2
    assert pa.decode_path(params(max_seq_len=4096, v1_max_seq_len=2048)) == 2
    assert pa.decode_path(params(max_seq_len=4096, v1_max_seq_len=4096)) == 1
    assert pa.decode_path(params(num_kv_heads=7)) == 0


def test_decode_launches(L):
    """pa_decode_launches: V1 is one launch; V2 is one launch where the
    tensor-core kernel runs a persistent grid with a CTA per reduce unit (one
    100K-token sequence, 24 heads), else two; invalid parameters and empty
    batches make none."""
    assert L.pa_decode_launches(ctypes.byref(params(max_seq_len=8192))) == 1
    assert L.pa_decode_launches(ctypes.byref(params(num_heads=25))) == 0
    assert L.pa_decode_launches(ctypes.byref(params(num_seqs=0))) == 0
    v2 = L.pa_decode_launches(ctypes.byref(params()))
    assert v2 == (1 if pa.decode_kernel(params()) == 2 else 2)
    # the CUDA-core path keeps the dependent reduce kernel
    assert L.pa_decode_launches(ctypes.byref(params(flags=pa.PA_FLAG_PORTABLE))) == 2
    # more reduce units (32 rows x 8 slices of 32) than the persistent grid's CTAs
    big = params(num_seqs=32, max_blocks_per_seq=6250)
    assert L.pa_decode_launches(ctypes.byref(big)) == 2


def test_status_strings(L):
    for code in range(0, 10):
        s = pa.status_string(code)
        assert s and s != "unknown status"
    assert pa.status_string(99) == "unknown status"


def _call_v2(L, p, q=256, k=256, v=256, bt=256, sl=256, ws=256, ws_bytes=1 << 40, out=256):
    V = ctypes.c_void_p
    return L.pa_decode_v2(ctypes.byref(p), V(q), V(k), V(v), V(bt), V(sl), V(ws), ws_bytes, V(out),
                          V(0))


def _call_v1(L, p, q=256, k=256, v=256, bt=256, sl=256, out=256):
    V = ctypes.c_void_p
    return L.pa_decode_v1(ctypes.byref(p), V(q), V(k), V(v), V(bt), V(sl), V(out), V(0))


# Each case fails a host check, so nothing is launched (the fake addresses are
# never dereferenced).
def test_host_checks_reject_bad_arguments(L):
    assert _call_v2(L, params(), q=0) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(), out=0) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(), ws=0) == pa.PA_ERR_INVALID_ARG
    assert _call_v1(L, params(), bt=0) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(), q=264) == pa.PA_ERR_MISALIGNED      # 8-byte aligned only
    assert _call_v2(L, params(), k=258) == pa.PA_ERR_MISALIGNED
    assert _call_v2(L, params(), sl=258) == pa.PA_ERR_MISALIGNED
    assert _call_v2(L, params(), ws=272) == pa.PA_ERR_MISALIGNED     # not 256-byte aligned
    assert _call_v2(L, params(), ws_bytes=1000) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    assert _call_v2(L, params(num_kv_heads=5)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(partition_size=24)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(partition_size=0)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(head_dim=96)) == pa.PA_ERR_UNSUPPORTED
    assert _call_v2(L, params(kv_dtype=7)) == pa.PA_ERR_UNSUPPORTED
    assert _call_v2(L, params(out_dtype=pa.PA_F16)) == pa.PA_ERR_UNSUPPORTED   # bf16 kv
    assert _call_v2(L, params(max_seq_len=-1)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(max_seq_len=100001, max_blocks_per_seq=6250)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(num_blocks=0)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(flags=8)) == pa.PA_ERR_INVALID_ARG
    assert _call_v2(L, params(flags=16)) == pa.PA_ERR_INVALID_ARG
    # the split-x cache layout is a valid flag: the call gets past the
    # parameter checks and fails only on the undersized workspace
    assert _call_v2(L, params(flags=pa.PA_FLAG_SPLIT_X), ws_bytes=1000) == \
        pa.PA_ERR_WORKSPACE_TOO_SMALL
    assert pa.decode_kernel(params(flags=pa.PA_FLAG_SPLIT_X)) == 1   # CUDA-core kernels only
    assert L.pa_decode_v2(None, None, None, None, None, None, None, 0, None, None) == \
        pa.PA_ERR_INVALID_ARG
    V = ctypes.c_void_p
    p = params()
    assert L.pa_decode_v2_partitions(ctypes.byref(p), V(256), V(256), V(256), V(256), V(256),
                                     V(256), 1000, V(0)) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    assert L.pa_decode_v2_reduce(ctypes.byref(p), V(256), V(256), 1000, V(256), V(0)) == \
        pa.PA_ERR_WORKSPACE_TOO_SMALL
    assert L.pa_decode_v2_reduce(ctypes.byref(p), V(0), V(256), 1 << 40, V(256), V(0)) == \
        pa.PA_ERR_INVALID_ARG
    assert L.pa_decode_v2_reduce(ctypes.byref(p), V(256), V(256), 1 << 40, V(264), V(0)) == \
        pa.PA_ERR_MISALIGNED


def test_empty_batch_is_a_no_op(L):
    # num_seqs == 0: nothing to do, no pointer is looked at
    assert _call_v2(L, params(num_seqs=0), q=0, k=0, v=0, bt=0, sl=0, ws=0, out=0) == pa.PA_OK
    assert _call_v1(L, params(num_seqs=0), q=0, k=0, v=0, bt=0, sl=0, out=0) == pa.PA_OK


def test_workspace_helpers_check_arguments(L):
    V = ctypes.c_void_p
    assert L.pa_workspace_init(V(0), 1024, V(0)) == pa.PA_ERR_INVALID_ARG
    assert L.pa_workspace_init(V(272), 1024, V(0)) == pa.PA_ERR_MISALIGNED
    v = ctypes.c_int32(0)
    assert L.pa_read_device_status(V(0), ctypes.byref(v), 0, V(0)) == pa.PA_ERR_INVALID_ARG
    assert L.pa_version() >= 100


def test_decode_kernel_query(L):
    # 0 for invalid parameters; the CUDA-core family whenever asked for, or
    # for float32 caches; otherwise whatever the device supports
    assert pa.decode_kernel(params(num_kv_heads=5)) == 0
    assert pa.decode_kernel(params(flags=pa.PA_FLAG_PORTABLE)) == 1
    assert pa.decode_kernel(params(kv_dtype=pa.PA_F32)) == 1
    assert pa.decode_kernel(params(num_heads=36, num_kv_heads=4)) == 1   # group 9 > 8
    assert pa.decode_kernel(params()) in (1, 2)


def test_host_staging_size_and_checks(L):
    """pa_host_staging_size: q | block_tables | seq_lens | out, each rounded to
    256 bytes; pa_decode_host refuses a missing, misaligned or short staging
    buffer before it enqueues anything."""
    r = lambda x: (x + 255) // 256 * 256
    p = params(num_seqs=2, max_blocks_per_seq=6250)
    want = r(2 * 24 * 256 * 2) + r(2 * 6250 * 4) + r(2 * 4) + r(2 * 24 * 256 * 4)
    assert pa.host_staging_size(p) == want
    assert pa.host_staging_size(params(num_heads=25)) == 0          # invalid parameters
    fake = ctypes.c_void_p(0x10000)                                   # never dereferenced
    call = lambda staging, nbytes: L.pa_decode_host(ctypes.byref(p), fake, fake, fake, fake, fake,
                                                    fake, 1 << 30, staging, nbytes, fake, None)
    assert call(None, want) == pa.PA_ERR_INVALID_ARG
    assert call(ctypes.c_void_p(0x10008), want) == pa.PA_ERR_MISALIGNED
    assert call(ctypes.c_void_p(0x10000), want - 1) == pa.PA_ERR_WORKSPACE_TOO_SMALL
    # misaligned caches are refused before the host-to-device copies are queued
    odd = ctypes.c_void_p(0x10008)
    for k, v in ((odd, fake), (fake, odd)):
        assert L.pa_decode_host(ctypes.byref(p), fake, k, v, fake, fake, fake, 1 << 30,
                                ctypes.c_void_p(0x10000), want, fake, None) == \
            pa.PA_ERR_MISALIGNED
    # the offsets of the same layout (for a host mirror of it)
    off = pa.host_staging_offsets(p)
    assert off == (0, r(2 * 24 * 256 * 2), r(2 * 24 * 256 * 2) + r(2 * 6250 * 4),
                   r(2 * 24 * 256 * 2) + r(2 * 6250 * 4) + r(2 * 4), want)
    assert L.pa_host_staging_offsets(ctypes.byref(p), None) == pa.PA_ERR_INVALID_ARG
    bad = (ctypes.c_size_t * 5)()
    assert L.pa_host_staging_offsets(ctypes.byref(params(num_heads=25)), bad) == \
        pa.PA_ERR_INVALID_ARG
