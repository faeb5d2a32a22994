"""Helpers for the GPU parity tests: run the CUDA path through the Python
binding (which calls the C ABI) and measure its distance to the oracle."""
from __future__ import annotations

import numpy as np
import torch

# Tolerance for attention outputs against the fp64 oracle on N(0,1) inputs.
MAX_ABS = 5e-3
REL_L2 = 2e-3


def fa():
    import causal_gqa_flash_attn_gb300 as m
    m.lib()
    return m


def errors(got, want):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    d = got - want
    return float(np.max(np.abs(d))) if d.size else 0.0, float(
        np.linalg.norm(d) / max(np.linalg.norm(want), 1e-300))


def assert_close(got, want, what=""):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    ma, rl = errors(got, want)
    assert ma <= MAX_ABS and rl <= REL_L2, f"{what}: max_abs={ma:.3e} rel_l2={rl:.3e}"
    return ma, rl


def fmt_code(kv_fmt: str) -> int:
    from workloads import FMT_CODES
    return FMT_CODES[kv_fmt]


def build_cache(k, v, *, kv_fmt, shadow_sink=0, shadow_win=0, max_seq=None, pos0=None,
                k_scale=1.0, v_scale=1.0):
    """Append K, V ([nslots][n][Hkv][hd] or [n][Hkv][hd] float32 numpy) into
    fresh planes (fp8 planes with the given scales); returns (k_planes,
    v_planes, max_seq)."""
    m = fa()
    k = np.asarray(k, np.float32)
    v = np.asarray(v, np.float32)
    if k.ndim == 3:
        k, v = k[None], v[None]
    nslots, n, hkv, hd = k.shape
    if max_seq is None:
        max_seq = n
    code = fmt_code(kv_fmt)
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=k_scale)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=v_scale)
    p0 = torch.zeros(nslots, dtype=torch.int32, device="cuda") if pos0 is None else \
        torch.as_tensor(np.asarray(pos0, np.int32), device="cuda")
    m.kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kp, vp, p0,
                n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code,
                shadow_sink=shadow_sink, shadow_win=shadow_win)
    return kp, vp, max_seq


def run_prefill(q, k, v, *, kv_fmt, sink, win, shadow_sink=0, shadow_win=0, tile_map=False,
                max_seq=None, k_scale=1.0, v_scale=1.0):
    """Append then prefill on the GPU; returns out (numpy) and the tile map."""
    m = fa()
    n, hq, hd = q.shape
    hkv = k.shape[1]
    kp, vp, max_seq = build_cache(k, v, kv_fmt=kv_fmt, shadow_sink=shadow_sink,
                                  shadow_win=shadow_win, max_seq=max_seq, k_scale=k_scale,
                                  v_scale=v_scale)
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    out = torch.full((n, hq, hd), float("nan"), dtype=torch.float32, device="cuda")
    ws = torch.empty(m.prefill_workspace_bytes(n, hq, hkv, hd, kv_fmt=fmt_code(kv_fmt),
                                               shadow_win=shadow_win),
                     dtype=torch.uint8, device="cuda")
    tm = None
    if tile_map:
        bq, bk = m.prefill_tile_shape(hd)
        tm = torch.zeros((-(-n // bq)) * (-(-n // bk)), dtype=torch.uint8, device="cuda")
    m.prefill(qd, kp, vp, out, n, hq, hkv, hd, sink, win, fmt_code(kv_fmt), max_seq=max_seq,
              shadow_sink=shadow_sink, shadow_win=shadow_win, workspace=ws, tile_map=tm)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    res = out.cpu().numpy()
    if tile_map:
        return res, tm.cpu().numpy().reshape(-(-n // bq), -(-n // bk))
    return res


def run_decode(q, kp, vp, pos, *, hkv, hd, max_seq, sink, win, kv_fmt, shadow_sink=0,
               shadow_win=0, split_keys=256, max_splits=None):
    """fa_decode + fa_decode_combine; q [nslots][Hq][hd] numpy; returns out numpy."""
    m = fa()
    nslots, hq, _ = q.shape
    if max_splits is None:
        max_splits = max(1, -(-max_seq // split_keys))
    ws = torch.empty(m.decode_workspace_bytes(nslots, hq, hd, max_splits), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((nslots, hq, hd), float("nan"), dtype=torch.float32, device="cuda")
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    pd = torch.as_tensor(np.asarray(pos, np.int32), device="cuda")
    m.decode(qd, kp, vp, pd, n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq,
             sink=sink, win=win, kv_fmt=fmt_code(kv_fmt), shadow_sink=shadow_sink,
             shadow_win=shadow_win, split_keys=split_keys, max_splits=max_splits, workspace=ws)
    m.decode_combine(ws, out, nslots=nslots, n_q_heads=hq, head_dim=hd, max_splits=max_splits)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    return out.cpu().numpy()
