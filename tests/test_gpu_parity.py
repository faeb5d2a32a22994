"""Parity of the CUDA path (through the C ABI) with the CPU oracle.

Q4_0 bytes, fp16 shadow bytes and the prefill tile map must be bit-exact;
attention outputs must be within max-abs 5e-3 and relative L2 2e-3 of the
fp64 oracle on N(0,1) inputs."""

import numpy as np
import pytest
import torch

from conftest import golden_lines
from gpu_util import (assert_close, build_cache, fa, fmt_code, run_decode, run_prefill)
from workloads import decode_slot_inputs, prefill_inputs

pytestmark = pytest.mark.gpu

RNG_SEED = 4242


def plane_parts(planes, nslots, kv_fmt, hkv, max_seq, hd):
    """Split a planes tensor into per-slot (body, sink, ring) numpy views."""
    m = fa()
    code = fmt_code(kv_fmt)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    row, body_off, sink_off, ring_off = m.kv_plane_layout(code, hkv, max_seq, hd)
    raw = planes.cpu().numpy().reshape(nslots, pb)
    out = []
    for u in range(nslots):
        body = raw[u, body_off:body_off + hkv * max_seq * row].reshape(hkv, max_seq, row)
        if code == 1:
            sink = raw[u, sink_off:sink_off + hkv * 8 * hd * 2].view(np.uint16).reshape(hkv, 8, hd)
            ring = raw[u, ring_off:ring_off + hkv * 256 * hd * 2].view(np.uint16).reshape(hkv, 256, hd)
        else:
            sink = ring = None
        out.append((body, sink, ring))
    return out


# ------------------------------------------------------------------ append

@pytest.mark.parametrize("hd", [64, 128, 256])
def test_append_q4_bitexact(oracle_mod, hd):
    rng = np.random.default_rng(RNG_SEED + hd)
    nslots, n, hkv, max_seq = 3, 300, 2, 700
    k = rng.standard_normal((nslots, n, hkv, hd)).astype(np.float32)
    v = (rng.standard_normal((nslots, n, hkv, hd)) * 3).astype(np.float32)
    # special blocks from the hand-derived vectors, placed in row 5 of slot 1
    specials = [np.array([float(np.frombuffer(bytes.fromhex(t)[::-1], np.float32)[0])
                          for t in xs.split()], np.float32)
                for _, xs, _ in golden_lines("q4_encode.txt")]
    for i, sv in enumerate(specials[: hd // 32]):
        k[1, 5, 0, 32 * i:32 * i + 32] = sv
    pos0 = np.array([0, 7, 400], np.int32)
    kp, vp, _ = build_cache(k, v, kv_fmt="q4_0", shadow_sink=4, shadow_win=256,
                            max_seq=max_seq, pos0=pos0)
    for name, x, planes in (("K", k, kp), ("V", v, vp)):
        parts = plane_parts(planes, nslots, "q4_0", hkv, max_seq, hd)
        for u in range(nslots):
            body, sink, ring = parts[u]
            want = oracle_mod.q4_encode(x[u]).transpose(1, 0, 2)  # [hkv][n][row]
            p0 = pos0[u]
            assert np.array_equal(body[:, p0:p0 + n], want), (name, u)
            assert not body[:, :p0].any() and not body[:, p0 + n:].any()
            f16 = oracle_mod.f16_rne(x[u]).transpose(1, 0, 2)   # [hkv][n][hd]
            for s in range(4):
                if p0 <= s < p0 + n:
                    assert np.array_equal(sink[:, s], f16[:, s - p0]), (name, u, s)
            for t in range(max(0, n - 256), n):
                assert np.array_equal(ring[:, (p0 + t) % 256], f16[:, t]), (name, u, t)


def test_append_f32_copy():
    rng = np.random.default_rng(RNG_SEED)
    nslots, n, hkv, hd, max_seq = 2, 50, 2, 128, 120
    k = rng.standard_normal((nslots, n, hkv, hd)).astype(np.float32)
    v = rng.standard_normal((nslots, n, hkv, hd)).astype(np.float32)
    pos0 = np.array([3, 70], np.int32)
    kp, vp, _ = build_cache(k, v, kv_fmt="f32", max_seq=max_seq, pos0=pos0)
    for x, planes in ((k, kp), (v, vp)):
        parts = plane_parts(planes, nslots, "f32", hkv, max_seq, hd)
        for u in range(nslots):
            body = parts[u][0].view(np.float32)[:, :, :hd]
            assert np.array_equal(body[:, pos0[u]:pos0[u] + n], x[u].transpose(1, 0, 2))


def test_append_out_of_range_flags_device_error():
    m = fa()
    k = torch.zeros((1, 10, 2, 64), device="cuda")
    kp = m.alloc_planes(1, 1, 2, 16, 64)
    vp = m.alloc_planes(1, 1, 2, 16, 64)
    pos0 = torch.tensor([12], dtype=torch.int32, device="cuda")     # 12 + 10 > 16
    m.kv_append(k, k, kp, vp, pos0, n_kv_heads=2, head_dim=64, max_seq=16, kv_fmt=1)
    assert m.get_device_error() == m.ERR_DEVICE
    assert m.get_device_error() == m.OK                               # cleared
    body = plane_parts(kp, 1, "q4_0", 2, 16, 64)[0][0]
    assert body[:, 12:16].any() and not body[:, :12].any()           # in-range rows written


# ----------------------------------------------------------------- prefill

PREFILL_CASES = [
    # n, hq, hkv, hd, sink, win, fmt, shadow
    (1, 8, 2, 64, 0, 0, "f32", (0, 0)),
    (2, 4, 4, 64, 0, 0, "f32", (0, 0)),
    (15, 8, 1, 128, 0, 0, "f32", (0, 0)),
    (16, 16, 1, 256, 0, 1, "f32", (0, 0)),
    (17, 8, 2, 64, 4, 0, "f32", (0, 0)),
    (127, 8, 2, 64, 4, 16, "f32", (0, 0)),
    (128, 8, 2, 64, 0, 0, "f32", (0, 0)),
    (129, 4, 2, 128, 9, 3, "f32", (0, 0)),
    (300, 16, 2, 256, 4, 100, "f32", (0, 0)),
    (300, 2, 1, 256, 0, 300, "f32", (0, 0)),
    (300, 3, 3, 256, 4, 100, "f32", (0, 0)),
    (1000, 8, 1, 128, 4, 1024, "f32", (0, 0)),
    (700, 16, 2, 256, 0, 0, "f32", (0, 0)),
    (520, 16, 2, 256, 0, 0, "q4_0", (0, 0)),
    (520, 16, 2, 256, 0, 0, "q4_0", (4, 0)),
    (520, 16, 2, 256, 0, 0, "q4_0", (4, 256)),
    (400, 8, 2, 64, 4, 1, "q4_0", (8, 256)),
    (257, 4, 1, 128, 2, 40, "q4_0", (4, 256)),
    (100, 16, 1, 64, 0, 0, "q4_0", (8, 256)),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_small(oracle_mod, case):
    n, hq, hkv, hd, sink, win, fmt, (ss, sw) = case
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=RNG_SEED + n + hd)
    got = run_prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss, shadow_win=sw)
    want = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss,
                              shadow_win=sw)
    assert_close(got, want, str(case))


@pytest.mark.parametrize("hd", [64, 256])
@pytest.mark.parametrize("n,sink,win", [(1, 0, 0), (130, 0, 0), (600, 4, 1), (600, 4, 130),
                                        (1000, 0, 256), (1000, 200, 129), (777, 9, 3)])
def test_prefill_tile_map_bitexact(oracle_mod, n, sink, win, hd):
    q, k, v = prefill_inputs(n, 2, 1, hd, seed=RNG_SEED + 7)
    _, tm = run_prefill(q, k, v, kv_fmt="f32", sink=sink, win=win, tile_map=True)
    bq, bk = fa().prefill_tile_shape(hd)
    assert np.array_equal(tm, oracle_mod.tile_map(n, bq, bk, sink, win))


def test_prefill_deterministic():
    q, k, v = prefill_inputs(700, 16, 2, 256, seed=RNG_SEED)
    a = run_prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
    b = run_prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ decode

DECODE_CASES = [
    # lens per slot, hq, hkv, hd, sink, win, fmt, shadow, split_keys, max_seq
    ((1, 17, 300, 1000), 16, 2, 256, 4, 0, "q4_0", (4, 0), 256, 1024),
    ((513, 2000), 16, 2, 256, 0, 0, "q4_0", (4, 256), 256, 2048),
    ((700, 64, 1500), 8, 2, 128, 4, 100, "q4_0", (2, 64), 64, 1600),
    ((999, 5), 8, 1, 64, 0, 0, "f32", (0, 0), 100, 1000),
    ((1234,), 16, 1, 256, 3, 17, "f32", (0, 0), 256, 1300),
    ((640, 640, 640, 640), 4, 4, 64, 0, 0, "q4_0", (8, 256), 256, 700),
    # no window and no shadow window (the Q4_0 tiles are one run), including
    # slots whose every key is an fp16 sink (lengths 3 and 5 <= 8 sinks)
    ((3, 9, 40, 777), 8, 2, 128, 0, 0, "q4_0", (8, 0), 256, 800),
    ((5, 1300), 4, 1, 64, 2, 0, "q4_0", (8, 0), 128, 1400),
    # more tiles than body blocks, so that blocks run pieces of two or more
    # (slot, kv head) pairs one after another; with a window and shadows too
    ((4000, 3001, 2500, 17), 16, 2, 128, 4, 0, "q4_0", (4, 0), 256, 4096),
    ((6000, 5000, 33), 8, 2, 256, 4, 1024, "q4_0", (4, 256), 256, 6144),
    ((9000, 9000), 8, 1, 64, 0, 0, "q4_0", (0, 0), 256, 9000),
    # group 16 over Q4_0 (the generic kernel): sinks, a recent fp16 ring, a
    # window, and a narrow shadow window
    ((1, 17, 300, 1000), 16, 1, 256, 4, 0, "q4_0", (4, 0), 256, 1024),
    ((513, 2000), 32, 2, 128, 0, 0, "q4_0", (4, 256), 256, 2048),
    ((700, 64, 1500), 16, 1, 64, 4, 100, "q4_0", (2, 64), 64, 1600),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "-".join(map(str, c[1:])))
def test_decode_small(oracle_mod, case):
    lens, hq, hkv, hd, sink, win, fmt, (ss, sw), kps, max_seq = case
    nslots = len(lens)
    Lmax = max(lens)
    ks, vs, qs = [], [], []
    for u in range(nslots):
        qu, ku, vu = decode_slot_inputs(Lmax, hq, hkv, hd, seed=RNG_SEED + 11, slot=u)
        qs.append(qu)
        ks.append(ku)
        vs.append(vu)
    k = np.stack(ks)
    v = np.stack(vs)
    q = np.stack(qs)
    # every slot's cache holds exactly rows 0..len-1: append slot by slot
    m = fa()
    code = fmt_code(fmt)
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    for u, L in enumerate(lens):
        m.kv_append(torch.from_numpy(k[u:u + 1, :L]).cuda(), torch.from_numpy(v[u:u + 1, :L]).cuda(),
                    kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code, shadow_sink=ss, shadow_win=sw)
    pos = np.array(lens, np.int32) - 1
    got = run_decode(q, kp, vp, pos, hkv=hkv, hd=hd, max_seq=max_seq, sink=sink, win=win,
                     kv_fmt=fmt, shadow_sink=ss, shadow_win=sw, split_keys=kps)
    for u, L in enumerate(lens):
        want = oracle_mod.decode(q[u], L - 1, k[u], v[u], kv_fmt=fmt, sink=sink, win=win,
                                 shadow_sink=ss, shadow_win=sw)
        assert_close(got[u], want, f"{case} slot {u}")


def test_decode_bad_position_flags_device_error():
    m = fa()
    hq, hkv, hd, max_seq = 8, 2, 64, 100
    kp = m.alloc_planes(2, 1, hkv, max_seq, hd)
    vp = m.alloc_planes(2, 1, hkv, max_seq, hd)
    q = torch.zeros((2, hq, hd), device="cuda")
    pos = torch.tensor([5, 100], dtype=torch.int32, device="cuda")   # 100 >= max_seq
    ws = torch.empty(m.decode_workspace_bytes(2, hq, hd, 4), dtype=torch.uint8, device="cuda")
    m.decode(q, kp, vp, pos, n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq,
             sink=0, win=0, kv_fmt=1, split_keys=32, max_splits=4, workspace=ws)
    assert m.get_device_error() == m.ERR_DEVICE


def test_decode_deterministic():
    lens = (900, 300)
    hq, hkv, hd, max_seq = 16, 2, 256, 1024
    m = fa()
    rng = np.random.default_rng(5)
    k = rng.standard_normal((2, max_seq, hkv, hd)).astype(np.float32)
    v = rng.standard_normal((2, max_seq, hkv, hd)).astype(np.float32)
    q = rng.standard_normal((2, hq, hd)).astype(np.float32)
    kp, vp, _ = build_cache(k, v, kv_fmt="q4_0", shadow_sink=4, max_seq=max_seq)
    pos = np.array(lens, np.int32)
    a = run_decode(q, kp, vp, pos, hkv=hkv, hd=hd, max_seq=max_seq, sink=4, win=0,
                   kv_fmt="q4_0", shadow_sink=4)
    b = run_decode(q, kp, vp, pos, hkv=hkv, hd=hd, max_seq=max_seq, sink=4, win=0,
                   kv_fmt="q4_0", shadow_sink=4)
    assert np.array_equal(a, b)


# ----------------------------------------------------------------- combine

def test_combine_on_oracle_partials(oracle_mod):
    """fa_decode_combine alone, fed partials the oracle computed (empty ones
    included), against the oracle's merge."""
    m = fa()
    rng = np.random.default_rng(17)
    nslots, hq, hkv, hd, max_splits = 3, 8, 2, 128, 6
    L = 400
    E = 5
    ws_bytes = m.decode_workspace_bytes(nslots, hq, hd, max_splits)
    heads = nslots * hq
    up = lambda x: (x + 255) // 256 * 256
    S = max_splits + 1        # entry stride of fa_decode's workspace
    m_arr = np.full((heads, S), -np.inf, np.float32)
    l_arr = np.zeros((heads, S), np.float32)
    acc = np.zeros((heads, S, hd), np.float32)
    want = np.zeros((nslots, hq, hd))
    for u in range(nslots):
        q, k, v = decode_slot_inputs(L, hq, hkv, hd, seed=3, slot=u)
        kk, vv = oracle_mod.KVValues(k, "f32"), oracle_mod.KVValues(v, "f32")
        bounds = [0, 37, 37, 200, 399, 400]     # entry 1 is empty
        parts = [oracle_mod.partial(q, L - 1, bounds[e], bounds[e + 1], kk, vv, sink=0, win=0)
                 for e in range(E)]
        for h in range(hq):
            for e in range(E):
                m_arr[u * hq + h, e] = parts[e][0][h]
                l_arr[u * hq + h, e] = parts[e][1][h]
                acc[u * hq + h, e] = parts[e][2][h]
            want[u, h] = oracle_mod.combine([p[0][h] for p in parts], [p[1][h] for p in parts],
                                            np.array([p[2][h] for p in parts]))
    buf = np.zeros(ws_bytes, np.uint8)
    buf[:20] = np.array([0x46414443, nslots, hq, hd, E], np.uint32).view(np.uint8)
    o_m = 256
    o_l = o_m + up(heads * S * 4)
    o_a = o_l + up(heads * S * 4)
    buf[o_m:o_m + m_arr.nbytes] = m_arr.view(np.uint8).ravel()
    buf[o_l:o_l + l_arr.nbytes] = l_arr.view(np.uint8).ravel()
    buf[o_a:o_a + acc.nbytes] = acc.view(np.uint8).ravel()
    ws = torch.from_numpy(buf).cuda()
    out = torch.full((nslots, hq, hd), float("nan"), device="cuda")
    m.decode_combine(ws, out, nslots=nslots, n_q_heads=hq, head_dim=hd, max_splits=max_splits)
    assert m.get_device_error() == m.OK
    # partials were rounded to fp32 before the merge: compare at fp32 resolution
    got = out.cpu().numpy()
    assert np.max(np.abs(got - want)) < 1e-5


def test_combine_rejects_foreign_workspace():
    m = fa()
    ws = torch.zeros(m.decode_workspace_bytes(1, 8, 64, 4), dtype=torch.uint8, device="cuda")
    out = torch.full((1, 8, 64), 7.0, device="cuda")
    m.decode_combine(ws, out, nslots=1, n_q_heads=8, head_dim=64, max_splits=4)
    assert m.get_device_error() == m.ERR_DEVICE
    assert torch.all(out == 7.0)
