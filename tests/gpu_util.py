"""Helpers for the GPU parity tests: run the CUDA path through the Python
binding (which calls the C ABI) and measure its distance to the oracle."""
from __future__ import annotations

import json
import os

import numpy as np
import torch

# Tolerance for attention outputs against the fp64 oracle on N(0,1) inputs.
MAX_ABS = 5e-3
REL_L2 = 2e-3

# Redzones and poison (the substitute for a memory checker). Every buffer the
# helpers hand to the library sits between two guards of GUARD_BYTES bytes of
# GUARD_BYTE, and check_guards() asserts they are intact after the call: a
# write outside a buffer fails the test. Outputs start as NaN and workspaces as
# 0xff bytes (NaN in fp32 and fp16), so a value the kernels should have written
# and did not, or scratch read before it was written, reaches the result.
GUARD_BYTES = 4096
GUARD_BYTE = 0xA5
POISON_BYTE = 0xFF


def guarded(shape, dtype, *, fill=None, fill_byte=None):
    """A CUDA tensor of `shape` inside a guarded allocation; its data starts
    GUARD_BYTES after the allocation's (so its alignment is the allocator's)."""
    shape = (shape,) if isinstance(shape, int) else tuple(shape)
    numel = int(np.prod(shape, dtype=np.int64))
    esz = torch.empty(0, dtype=dtype).element_size()
    g = GUARD_BYTES // esz
    raw = torch.empty(numel + 2 * g, dtype=dtype, device="cuda")
    raw.view(torch.uint8).fill_(GUARD_BYTE)
    t = raw[g:g + numel]
    if fill is not None:
        t.fill_(fill)
    elif fill_byte is not None:
        t.view(torch.uint8).fill_(fill_byte)
    return t.view(shape)


def is_guarded(t) -> bool:
    st = t.untyped_storage()
    lo = t.storage_offset() * t.element_size()
    return lo == GUARD_BYTES and st.nbytes() - lo - t.numel() * t.element_size() == GUARD_BYTES


def check_guards(*named):
    """named: (what, tensor) pairs from guarded(); asserts both guards intact."""
    for what, t in named:
        assert is_guarded(t), f"{what}: not a guarded buffer"
        st = t.untyped_storage()
        b = torch.empty(0, dtype=torch.uint8, device=t.device).set_(st, 0, (st.nbytes(),), (1,))
        hi = GUARD_BYTES + t.numel() * t.element_size()
        assert bool((b[:GUARD_BYTES] == GUARD_BYTE).all()), f"{what}: write below the buffer"
        assert bool((b[hi:] == GUARD_BYTE).all()), f"{what}: write past the end of the buffer"


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
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    planes = []
    for scale in (k_scale, v_scale):
        t = guarded(nslots * pb, torch.uint8, fill_byte=POISON_BYTE)
        m.kv_init(t, code, hkv, max_seq, hd)
        if code == m.KV_FP8_E4M3 and scale != 1.0:
            m.kv_set_scale(t, code, hkv, max_seq, hd, scale)
        planes.append(t)
    kp, vp = planes
    p0 = torch.zeros(nslots, dtype=torch.int32, device="cuda") if pos0 is None else \
        torch.as_tensor(np.asarray(pos0, np.int32), device="cuda")
    m.kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kp, vp, p0,
                n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code,
                shadow_sink=shadow_sink, shadow_win=shadow_win)
    check_guards(("k planes", kp), ("v planes", vp))
    return kp, vp, max_seq


def run_prefill(q, k, v, *, kv_fmt, sink, win, shadow_sink=0, shadow_win=0, tile_map=False,
                max_seq=None, k_scale=1.0, v_scale=1.0, lse=False):
    """Append then prefill on the GPU (fa_prefill, or fa_prefill_lse with
    lse); returns out (numpy), then lse [Hq][n] with lse, then the tile map
    with tile_map."""
    m = fa()
    n, hq, hd = q.shape
    hkv = k.shape[1]
    kp, vp, max_seq = build_cache(k, v, kv_fmt=kv_fmt, shadow_sink=shadow_sink,
                                  shadow_win=shadow_win, max_seq=max_seq, k_scale=k_scale,
                                  v_scale=v_scale)
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    out = guarded((n, hq, hd), torch.float32, fill=float("nan"))
    ws = guarded(m.prefill_workspace_bytes(n, hq, hkv, hd, kv_fmt=fmt_code(kv_fmt),
                                           shadow_win=shadow_win),
                 torch.uint8, fill_byte=POISON_BYTE)
    tm = None
    if tile_map:
        bq, bk = m.prefill_tile_shape(hd)
        tm = guarded((-(-n // bq)) * (-(-n // bk)), torch.uint8, fill=0)
    lo = guarded((hq, n), torch.float32, fill=float("nan")) if lse else None
    m.prefill(qd, kp, vp, out, n, hq, hkv, hd, sink, win, fmt_code(kv_fmt), max_seq=max_seq,
              shadow_sink=shadow_sink, shadow_win=shadow_win, workspace=ws, tile_map=tm, lse=lo)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    check_guards(("out", out), ("workspace", ws), ("k planes", kp), ("v planes", vp),
                 *((("tile map", tm),) if tm is not None else ()),
                 *((("lse", lo),) if lo is not None else ()))
    res = [out.cpu().numpy()]
    if lse:
        res.append(lo.cpu().numpy())
    if tile_map:
        res.append(tm.cpu().numpy().reshape(-(-n // bq), -(-n // bk)))
    return res[0] if len(res) == 1 else tuple(res)


def run_chunk(q, k, v, pos0, *, hq, hkv, hd, sink, win, kv_fmt, shadow, want_map=False):
    """A cache filled as a caller continuing a sequence fills it (the context
    rows 0..pos0-1 in one append, the chunk's rows in a second), then
    fa_prefill_chunk with lse; returns out, lse [Hq][n] and the tile map."""
    m = fa()
    n = q.shape[0]
    L = pos0 + n
    code = fmt_code(kv_fmt)
    kp = m.alloc_planes(1, code, hkv, L, hd)
    vp = m.alloc_planes(1, code, hkv, L, hd)
    ss, sw = shadow
    for lo, hi in ((0, pos0), (pos0, L)):  # context, then the chunk
        if hi > lo:
            m.kv_append(torch.from_numpy(np.ascontiguousarray(k[None, lo:hi])).cuda(),
                        torch.from_numpy(np.ascontiguousarray(v[None, lo:hi])).cuda(), kp, vp,
                        torch.tensor([lo], dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                        head_dim=hd, max_seq=L, kv_fmt=code, shadow_sink=ss, shadow_win=sw)
    ws = guarded(m.prefill_chunk_workspace_bytes(pos0, n, hq, hkv, hd, kv_fmt=code,
                                                 shadow_win=sw),
                 torch.uint8, fill_byte=POISON_BYTE)
    out = guarded((n, hq, hd), torch.float32, fill=float("nan"))
    lse = guarded((hq, n), torch.float32, fill=float("nan"))
    tm = None
    if want_map:
        bq, bk = m.prefill_tile_shape(hd)
        tm = guarded((-(-n // bq), -(-L // bk)), torch.uint8, fill=0)
    m.prefill_chunk(torch.from_numpy(np.ascontiguousarray(q)).cuda(), kp, vp, out, pos0, n, hq,
                    hkv, hd, sink, win, code, max_seq=L, shadow_sink=ss, shadow_win=sw,
                    workspace=ws, tile_map=tm, lse=lse)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    check_guards(("out", out), ("lse", lse), ("workspace", ws),
                 *((("tile map", tm),) if tm is not None else ()))
    return out.cpu().numpy(), lse.cpu().numpy(), (tm.cpu().numpy() if want_map else None)


def record_parity(test, **values):
    """Append one JSON line of measured errors to the file named by the
    FA_PARITY_LOG environment variable (nothing when it is unset)."""
    path = os.environ.get("FA_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"test": test, **values}) + "\n")


def run_decode(q, kp, vp, pos, *, hkv, hd, max_seq, sink, win, kv_fmt, shadow_sink=0,
               shadow_win=0, split_keys=256, max_splits=None):
    """fa_decode + fa_decode_combine; q [nslots][Hq][hd] numpy; returns out numpy."""
    m = fa()
    nslots, hq, _ = q.shape
    if max_splits is None:
        max_splits = max(1, -(-max_seq // split_keys))
    ws = guarded(m.decode_workspace_bytes(nslots, hq, hd, max_splits), torch.uint8,
                 fill_byte=POISON_BYTE)
    out = guarded((nslots, hq, hd), torch.float32, fill=float("nan"))
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    pd = torch.as_tensor(np.asarray(pos, np.int32), device="cuda")
    m.decode(qd, kp, vp, pd, n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq,
             sink=sink, win=win, kv_fmt=fmt_code(kv_fmt), shadow_sink=shadow_sink,
             shadow_win=shadow_win, split_keys=split_keys, max_splits=max_splits, workspace=ws)
    m.decode_combine(ws, out, nslots=nslots, n_q_heads=hq, head_dim=hd, max_splits=max_splits)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    check_guards(("out", out), ("workspace", ws),
                 *((w, t) for w, t in (("k planes", kp), ("v planes", vp)) if is_guarded(t)))
    return out.cpu().numpy()
