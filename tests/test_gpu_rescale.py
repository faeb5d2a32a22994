"""Parity with the oracle on inputs that make the kernels rescale O.

The kernels keep O and the row sum l against a stale reference of the running
maximum and rescale them only when the maximum grows past a threshold (2^8 in
the prefill and the generic and dense decodes, 2^2 in the Q4_0 decode). On
N(0,1) inputs the maximum settles within the first key tiles, so that path
hardly runs. Here every query is u + 0.5 N(0,1) and key j is
a(j) u + N(0,1), with u the alternating +-1 vector and a(j) rising by one step
per 128 keys for the first four tiles: a query's scores rise by about 9 (in
the exp2 domain) from one of those tiles to the next, so the maximum passes
the threshold on each. The rise is spread over all head_dim terms, so every
operand stays O(1) and the fp16 operand rounding stays as small as on N(0,1)
inputs. Outputs are compared with the fp64 oracle at the usual tolerance
(max-abs 5e-3, relative L2 2e-3), the prefill's log-sum-exps within 5e-3."""

import numpy as np
import pytest
import torch

from gpu_util import assert_close, fa, fmt_code, run_chunk, run_decode, run_prefill
from workloads import decode_slot_inputs, prefill_inputs

pytestmark = pytest.mark.gpu

RISE_LOG2 = 9.0   # score rise per tile, exp2 domain
RISE_TILES = 4    # tiles over which the scores rise
SEED = 5150


def rising(q, k):
    """q and k (rows on the first axis of k, head_dim last) rebuilt as above."""
    hd = q.shape[-1]
    u = np.where(np.arange(hd) % 2 == 0, 1.0, -1.0).astype(np.float32)
    step = RISE_LOG2 / (np.log2(np.e) / np.sqrt(hd)) / hd  # per tile, per element of u
    q = (u + 0.5 * q).astype(np.float32)
    rows = np.arange(k.shape[0])
    a = (step * np.minimum(rows // 128, RISE_TILES)).astype(np.float32)
    k = (a.reshape((-1,) + (1,) * (k.ndim - 1)) * u + k).astype(np.float32)
    return q, k


# (n, hq, hkv, hd, sink, win, fmt, (shadow_sink, shadow_win), k_scale)
PREFILL_CASES = [
    (700, 16, 2, 256, 0, 0, "f32", (0, 0), 1.0),
    (700, 16, 2, 256, 4, 300, "f32", (0, 0), 1.0),
    (600, 8, 2, 64, 0, 0, "f32", (0, 0), 1.0),
    (520, 16, 2, 256, 0, 0, "q4_0", (4, 256), 1.0),
    (520, 16, 2, 256, 0, 0, "f16", (0, 0), 1.0),
    (520, 16, 2, 256, 0, 0, "fp8_e4m3", (0, 0), 16.0),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_rescales_every_tile(oracle_mod, case):
    n, hq, hkv, hd, sink, win, fmt, (ss, sw), ksc = case
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=SEED + n + hd)
    q, k = rising(q, k)
    got, got_lse = run_prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss,
                               shadow_win=sw, k_scale=ksc, lse=True)
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss,
                                        shadow_win=sw, k_scale=ksc, with_lse=True)
    assert_close(got, want, str(case))
    err = np.max(np.abs(got_lse - want_lse.T))
    assert np.all(np.isfinite(got_lse)) and err <= 5e-3, f"{case}: lse max-abs {err:.3g}"


@pytest.mark.parametrize("fmt,shadow", [("f32", (0, 0)), ("q4_0", (4, 64))])
def test_prefill_chunk_rescales_every_tile(oracle_mod, fmt, shadow):
    """The chunked prefill (with a shadow window narrower than the ring, its
    two merged parts) on rising scores."""
    pos0, n, hq, hkv, hd, sink, win = 300, 400, 16, 2, 256, 4, 256
    L = pos0 + n
    q_all, k, v = prefill_inputs(L, hq, hkv, hd, seed=SEED + 1)
    q_all, k = rising(q_all, k)
    q = q_all[pos0:]
    out, lse, _ = run_chunk(q, k, v, pos0, hq=hq, hkv=hkv, hd=hd, sink=sink, win=win,
                            kv_fmt=fmt, shadow=shadow)
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win,
                                        shadow_sink=shadow[0], shadow_win=shadow[1],
                                        with_lse=True, pos0=pos0)
    assert_close(out, want, f"{fmt} {shadow}")
    err = np.max(np.abs(lse - want_lse.T))
    assert np.all(np.isfinite(lse)) and err <= 5e-3, f"{fmt} {shadow}: lse max-abs {err:.3g}"


# (lens, hq, hkv, hd, sink, win, fmt, (shadow_sink, shadow_win), split_keys, max_seq, k_scale)
DECODE_CASES = [
    ((3000, 1500), 16, 2, 256, 0, 0, "f32", (0, 0), 1024, 3072, 1.0),
    ((3000, 1500), 16, 2, 256, 4, 1000, "q4_0", (4, 256), 1024, 3072, 1.0),
    ((3000, 1500), 16, 1, 256, 0, 0, "q4_0", (0, 0), 1024, 3072, 1.0),
    ((3000, 1500), 16, 2, 256, 0, 0, "f16", (0, 0), 1024, 3072, 1.0),
    ((3000, 1500), 16, 2, 256, 0, 0, "fp8_e4m3", (0, 0), 1024, 3072, 32.0),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "-".join(map(str, c[1:])))
def test_decode_rescales_every_tile(oracle_mod, case):
    lens, hq, hkv, hd, sink, win, fmt, (ss, sw), kps, max_seq, ksc = case
    m = fa()
    code = fmt_code(fmt)
    nslots = len(lens)
    qs, ks, vs = [], [], []
    for u in range(nslots):
        qu, ku, vu = decode_slot_inputs(max(lens), hq, hkv, hd, seed=SEED + 7, slot=u)
        qu, ku = rising(qu, ku)
        qs.append(qu)
        ks.append(ku)
        vs.append(vu)
    q = np.stack(qs)
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=ksc)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=1.0)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    for u, L in enumerate(lens):
        m.kv_append(torch.from_numpy(ks[u][None, :L]).cuda(),
                    torch.from_numpy(vs[u][None, :L]).cuda(), kp[u * pb:(u + 1) * pb],
                    vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code, shadow_sink=ss, shadow_win=sw)
    pos = np.array(lens, np.int32) - 1
    got = run_decode(q, kp, vp, pos, hkv=hkv, hd=hd, max_seq=max_seq, sink=sink, win=win,
                     kv_fmt=fmt, shadow_sink=ss, shadow_win=sw, split_keys=kps)
    for u, L in enumerate(lens):
        want = oracle_mod.decode(q[u], L - 1, ks[u], vs[u], kv_fmt=fmt, sink=sink, win=win,
                                 shadow_sink=ss, shadow_win=sw, k_scale=ksc)
        assert_close(got[u], want, f"{case} slot {u}")
