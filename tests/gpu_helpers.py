"""Helpers for the GPU parity tests: run the CUDA path through the binding and
compare with the float64 oracle."""
from __future__ import annotations

import numpy as np
import torch

import paged_attention_decode_v2_gb300 as pa

TOL = {torch.float32: 1e-5, torch.bfloat16: 2e-3, torch.float16: 2e-3}


CONTROL_BYTES = 1024        # the workspace's control block (status, marker, counters)
GUARD_BYTES = 4096          # canary region on each side of out and the workspace
GUARD_F = -4096.0           # canary of out's guards (exact in f32, bf16 and f16)
GUARD_B = 0xA5              # canary byte of the workspace's guards


def _guarded(n_elems, dtype, fill, device):
    """A tensor of n_elems elements with GUARD_BYTES of canaries on each side
    (the interior stays 256-byte aligned): returns (whole, interior)."""
    esz = torch.tensor([], dtype=dtype).element_size()
    g = GUARD_BYTES // esz
    whole = torch.empty(n_elems + 2 * g, dtype=dtype, device=device)
    whole.fill_(fill)
    return whole, whole[g:g + n_elems]


def _guards_intact(whole, n_elems, fill):
    g = GUARD_BYTES // whole.element_size()
    lo, hi = whole[:g], whole[g + n_elems:]
    return bool((lo == fill).all().item()) and bool((hi == fill).all().item())


def split_x_caches(batch):
    """The caches of ``batch`` rewritten (as test input, on the batch's
    device) into the split-x layout: keys [blocks, kv_heads, head_dim / x,
    block_size, x], values [blocks, kv_heads, head_dim, block_size],
    x = 16 / element bytes."""
    nb, hkv, bs, d = batch.k_cache.shape
    x = 16 // batch.k_cache.element_size()
    k5 = batch.k_cache.view(nb, hkv, bs, d // x, x).permute(0, 1, 3, 2, 4).contiguous()
    v4 = batch.v_cache.permute(0, 1, 3, 2).contiguous()
    return k5, v4


def run(batch, path="decode", partition_size=512, portable=False, out_dtype=torch.float32,
        v1_max_seq_len=pa.DEFAULT_V1_MAX_SEQ_LEN, workspace=None, return_ws=False,
        check_status=True, split_x=False):
    """Run one decode step of ``batch`` (already on the GPU); returns out as a
    float64 numpy array (and the workspace tensor when asked).  When a
    workspace was used, its device status word must read OK afterwards
    (unless ``check_status`` is False).  ``out`` and a workspace made here
    sit between canary regions that must be untouched after the call (no
    write outside the buffers the call was given).  ``split_x``: the caches
    go in rewritten into the split-x layout."""
    b = batch
    kc, vc = split_x_caches(b) if split_x else (b.k_cache, b.v_cache)
    n_out = int(np.prod(tuple(b.q.shape)))
    out_whole, out_flat = _guarded(n_out, out_dtype, GUARD_F, b.q.device)
    out_flat.fill_(float("nan"))
    out = out_flat.view(tuple(b.q.shape))
    params = pa.make_params(b.q, kc, b.block_tables, max_seq_len=b.max_seq_len,
                            scale=b.scale, partition_size=partition_size, out_dtype=out_dtype,
                            v1_max_seq_len=v1_max_seq_len, portable=portable, split_x=split_x)
    ws_whole = None
    if workspace is None and path in ("v2", "decode"):
        n = pa.workspace_size(params)
        ws_whole, workspace = _guarded(n, torch.uint8, GUARD_B, b.q.device)
        workspace.view(torch.float32).fill_(float("nan"))        # poison everything,
        pa.workspace_init(workspace)                              # then the control block
    kw = dict(max_seq_len=b.max_seq_len, scale=b.scale, portable=portable, split_x=split_x)
    if path == "v1":
        pa.decode_v1(b.q, kc, vc, b.block_tables, b.seq_lens, out, **kw)
    elif path == "v2":
        pa.decode_v2(b.q, kc, vc, b.block_tables, b.seq_lens, out, workspace,
                     partition_size=partition_size, **kw)
    else:
        pa.decode(b.q, kc, vc, b.block_tables, b.seq_lens, out, workspace,
                  partition_size=partition_size, v1_max_seq_len=v1_max_seq_len, **kw)
    torch.cuda.synchronize()
    assert _guards_intact(out_whole, n_out, GUARD_F), "write outside out"
    if ws_whole is not None:
        assert _guards_intact(ws_whole, workspace.numel(), GUARD_B), "write outside the workspace"
    if check_status and workspace is not None and path in ("v2", "decode"):
        st = pa.read_device_status(workspace, clear=False)
        assert st == pa.PA_OK, f"device status {st}: {pa.status_string(st)}"
    res = out.double().cpu().numpy()
    return (res, workspace) if return_ws else res


def max_err(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    if a.size == 0:
        return 0.0
    return float(np.max(np.abs(a - b)))


def assert_close(gpu, ref, tol, what=""):
    gpu = np.asarray(gpu)
    assert np.all(np.isfinite(gpu)), f"{what}: non-finite output"
    err = max_err(gpu, ref)
    assert err <= tol, f"{what}: max abs err {err:.3e} > {tol:.1e}"
    return err


def bf16_round(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def workspace_views(ws, batch, partition_size):
    """max_logits, exp_sums, tmp_out views of a V2 workspace (layout of pa.h)."""
    w = batch.workload
    B, H, D = w.num_seqs, w.num_heads, w.head_dim
    NP = max(1, -(-batch.max_seq_len // partition_size))
    r = lambda x: (x + 255) // 256 * 256
    f = ws.view(torch.float32)
    o_ml = CONTROL_BYTES
    o_es = o_ml + r(B * H * NP * 4)
    o_to = o_es + r(B * H * NP * 4)
    ml = f[o_ml // 4:o_ml // 4 + B * H * NP].view(B, H, NP)
    es = f[o_es // 4:o_es // 4 + B * H * NP].view(B, H, NP)
    to = f[o_to // 4:o_to // 4 + B * H * NP * D].view(B, H, NP, D)
    return ml.double().cpu().numpy(), es.double().cpu().numpy(), to.double().cpu().numpy()


def control_words(ws):
    """The control block's words: (marker, epoch, CTAs started, finished
    counters [2], unit queues [2]) of the one-launch V2 step."""
    w = ws[:CONTROL_BYTES].view(torch.int32).cpu().numpy().astype(np.int64) & 0xFFFFFFFF
    start = int(w[64]) | (int(w[65]) << 32)
    return int(w[1]), start >> 32, start & 0xFFFFFFFF, w[66:68].tolist(), w[68:70].tolist()


MARKER = 0x5A5A5A5A
