"""Parity with the oracle over seeded random shapes.

Each case is drawn once, at import, from a fixed seed: head_dim 64, 128 or
256, 1 to 3 kv heads with 1, 2, 4, 8 or 16 query heads each, ragged lengths,
sinks and windows (or none), every cache format, Q4_0 fp16 shadows of any
allowed size, fp8 planes with scales other than 1. Prefill cases append then
prefill one sequence; decode cases fill 1 to 5 slots of different lengths and
decode one query per slot. Outputs are compared with the fp64 oracle at the
usual tolerance (max-abs 5e-3, relative L2 2e-3)."""

import numpy as np
import pytest
import torch

from gpu_util import assert_close, build_cache, fa, fmt_code, run_decode, run_prefill
from workloads import decode_slot_inputs, prefill_inputs

pytestmark = pytest.mark.gpu

FORMATS = ("f32", "q4_0", "f16", "fp8_e4m3")


def _attention_mask(rng, longest):
    """(sink, win): no window half of the time, else a window of 1..longest+50
    and 0..10 sinks."""
    if rng.random() < 0.5:
        return 0, 0
    return int(rng.integers(0, 11)), int(rng.integers(1, longest + 51))


def _format(rng):
    fmt = FORMATS[int(rng.integers(0, len(FORMATS)))]
    ss = sw = 0
    ks = vs = 1.0
    if fmt == "q4_0":
        ss = int(rng.integers(0, 9))
        sw = int(rng.choice([0, 256, int(rng.integers(1, 257))]))
    if fmt == "fp8_e4m3":
        ks, vs = (float(x) for x in rng.uniform(0.5, 2.0, size=2))
    return fmt, ss, sw, ks, vs


def _heads(rng):
    hd = int(rng.choice([64, 128, 256]))
    hkv = int(rng.integers(1, 4))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    return hd, hkv * g, hkv


def _prefill_cases(count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(count):
        hd, hq, hkv = _heads(rng)
        n = int(rng.integers(1, 701))
        sink, win = _attention_mask(rng, n)
        out.append((n, hq, hkv, hd, sink, win) + _format(rng))
    return out


def _decode_cases(count, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    out = []
    for _ in range(count):
        hd, hq, hkv = _heads(rng)
        lens = tuple(int(x) for x in rng.integers(1, 3001, size=int(rng.integers(1, 6))))
        sink, win = _attention_mask(rng, max(lens))
        kps = int(rng.choice([64, 256, 1024]))
        max_seq = max(lens) + int(rng.integers(0, 100))
        out.append((lens, hq, hkv, hd, sink, win) + _format(rng) + (kps, max_seq))
    return out


PREFILL_CASES = _prefill_cases(24, 20261202)
DECODE_CASES = _decode_cases(16, 20261203)


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "-".join(map(str, c[:9])))
def test_prefill_random_shape(oracle_mod, case):
    n, hq, hkv, hd, sink, win, fmt, ss, sw, ks, vs = case
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=n * 7 + hq + hd)
    got = run_prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss, shadow_win=sw,
                      k_scale=ks, v_scale=vs)
    want = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss,
                              shadow_win=sw, k_scale=ks, v_scale=vs)
    assert_close(got, want, str(case))


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "-".join(map(str, c[1:9])))
def test_decode_random_shape(oracle_mod, case):
    lens, hq, hkv, hd, sink, win, fmt, ss, sw, ks, vs, kps, max_seq = case
    nslots = len(lens)
    qs, ksl, vsl = [], [], []
    for u in range(nslots):
        qu, ku, vu = decode_slot_inputs(max(lens), hq, hkv, hd, seed=sum(lens) + hd, slot=u)
        qs.append(qu)
        ksl.append(ku)
        vsl.append(vu)
    q = np.stack(qs)
    m = fa()
    code = fmt_code(fmt)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=ks)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=vs)
    for u, L in enumerate(lens):  # each slot's cache holds exactly its rows 0..L-1
        m.kv_append(torch.from_numpy(ksl[u][None, :L]).cuda(),
                    torch.from_numpy(vsl[u][None, :L]).cuda(), kp[u * pb:(u + 1) * pb],
                    vp[u * pb:(u + 1) * pb], torch.zeros(1, dtype=torch.int32, device="cuda"),
                    n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code, shadow_sink=ss,
                    shadow_win=sw)
    pos = np.array(lens, np.int32) - 1
    got = run_decode(q, kp, vp, pos, hkv=hkv, hd=hd, max_seq=max_seq, sink=sink, win=win,
                     kv_fmt=fmt, shadow_sink=ss, shadow_win=sw, split_keys=kps)
    for u, L in enumerate(lens):
        want = oracle_mod.decode(q[u], L - 1, ksl[u], vsl[u], kv_fmt=fmt, sink=sink, win=win,
                                 shadow_sink=ss, shadow_win=sw, k_scale=ks, v_scale=vs)
        assert_close(got[u], want, f"{case} slot {u}")
