"""Pins of the CPU oracle to facts the pages and the mathematics fix.

Nothing here compares the oracle with itself: each test checks it against a
hand-derived vector (tests/golden), a library routine (numpy's binary16
conversion, scipy's softmax), a closed form, or an invariant of attention
stated on the pages ("attention.cu" file header; "vt/ops.h" vt::Attention;
"attention.cu" "Decode-mode flash attention").
"""
import math
import struct

import numpy as np
import pytest
from scipy.special import softmax

from conftest import golden_lines


def f32_from_hex(h):
    return struct.unpack("<f", struct.pack("<I", int(h, 16)))[0]


# ------------------------------------------------------------------ fp16

def test_f16_golden(oracle_mod):
    for name, xb, hb in golden_lines("f16_rne.txt"):
        x = np.array([f32_from_hex(xb)], np.float32)
        assert int(oracle_mod.f16_rne(x)[0]) == int(hb, 16), name


def test_f16_matches_numpy_conversion(oracle_mod):
    """numpy's float32 -> float16 cast is an independent round-to-nearest-even."""
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=400000, dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32)
    x = x[~np.isnan(x)]
    # dense coverage of the fp16 range, ties included
    y = (np.arange(-70000, 70000, 0.03125, dtype=np.float64)).astype(np.float32)
    z = np.ldexp(rng.standard_normal(100000), rng.integers(-30, 17, 100000)).astype(np.float32)
    for arr in (x, y, z):
        with np.errstate(over="ignore"):
            ref = arr.astype(np.float16).view(np.uint16)
        assert np.array_equal(oracle_mod.f16_rne(arr), ref)


def test_f16_nan_stays_nan(oracle_mod):
    """A NaN becomes a binary16 NaN of the same sign (exponent all ones, mantissa
    not zero), and the canonical quiet NaN the value numpy's cast gives."""
    bits = np.array([0x7fc00000, 0xffc00000, 0x7f800001, 0xff800001, 0x7fffffff, 0x7fa00000],
                    dtype=np.uint32)
    h = oracle_mod.f16_rne(bits.view(np.float32)).astype(np.uint32)
    assert np.all((h & 0x7c00) == 0x7c00) and np.all((h & 0x03ff) != 0)
    assert np.array_equal(h >> 15, bits >> 31)
    ref = np.array([np.nan], np.float32).astype(np.float16).view(np.uint16)
    assert oracle_mod.f16_rne(np.array([np.nan], np.float32))[0] == ref[0]


def test_f16_decode_matches_numpy(oracle_mod):
    h = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    ref = h.view(np.float16).astype(np.float64)
    got = oracle_mod.f16_to_f64(h)
    finite = np.isfinite(ref)
    assert np.array_equal(got[finite], ref[finite])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


# ------------------------------------------------------------------ Q4_0

def test_q4_encode_golden(oracle_mod):
    for name, xs, bs in golden_lines("q4_encode.txt"):
        x = np.array([f32_from_hex(t) for t in xs.split()], np.float32)
        want = bytes(int(t, 16) for t in bs.split())
        got = oracle_mod.q4_encode(x[None, :])[0].tobytes()
        assert got == want, (name, got.hex(), want.hex())


def test_q4_decode_golden(oracle_mod):
    for name, bs, vs in golden_lines("q4_decode.txt"):
        b = np.array([int(t, 16) for t in bs.split()], np.uint8)
        want = np.array([float(t) for t in vs.split()])
        got = oracle_mod.q4_decode(b[None, :], 32)[0]
        assert np.array_equal(got, want), name


def test_q4_row_layout_is_blockwise(oracle_mod):
    """A row of head_dim values is head_dim/32 consecutive independent blocks."""
    rng = np.random.default_rng(3)
    x = rng.standard_normal((5, 256)).astype(np.float32)
    rows = oracle_mod.q4_encode(x)
    assert rows.shape == (5, 144)
    for r in range(5):
        for b in range(8):
            blk = oracle_mod.q4_encode(x[r:r + 1, 32 * b:32 * b + 32])[0]
            assert np.array_equal(rows[r, 18 * b:18 * b + 18], blk)


def test_q4_round_trip(oracle_mod):
    """decode then encode returns the same bytes when a code 0 element fixes
    amax = 8|d| and d is a normal fp16 (negative)."""
    rng = np.random.default_rng(11)
    for _ in range(2000):
        codes = rng.integers(0, 16, 32)
        codes[rng.integers(0, 32)] = 0
        e = rng.integers(-10, 10)
        d = -(1.0 + rng.integers(0, 1024) / 1024.0) * 2.0 ** e
        dh = np.array([d], np.float32).astype(np.float16).view(np.uint16)[0]
        b = np.zeros(18, np.uint8)
        b[0], b[1] = dh & 0xFF, dh >> 8
        for j in range(16):
            b[2 + j] = codes[j] | (codes[j + 16] << 4)
        x = oracle_mod.q4_decode(b[None], 32)[0].astype(np.float32)
        again = oracle_mod.q4_encode(x[None])[0]
        assert np.array_equal(again, b)


def test_q4_error_bound(oracle_mod):
    """|x - decode(encode(x))| <= |d| + 8 * 2^-11 * |d| (half a step from
    rounding, up to a full step on the clamped -amax side, plus the fp16
    rounding of d scaled by |c - 8| <= 8)."""
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((4000, 32)) * rng.uniform(0.01, 100, (4000, 1))).astype(np.float32)
    rec = oracle_mod.q4_decode(oracle_mod.q4_encode(x), 32)
    amax = np.abs(x.astype(np.float64)).max(axis=1, keepdims=True)
    d = amax / 8.0
    assert np.all(np.abs(x - rec) <= d * (1 + 8 * 2.0 ** -11) + 1e-30)


# ----------------------------------------------------------- visibility

def test_visible_rules(oracle_mod):
    V = oracle_mod.visible
    # win <= 0: full causal, sink ignored
    for p in range(20):
        for j in range(25):
            assert V(p, j, 7, 0) == (j <= p)
            assert V(p, j, 3, -5) == (j <= p)
    # a query always sees its own position (win >= 1)
    for p in range(40):
        for sink in range(0, 6):
            for win in range(1, 12):
                assert V(p, p, sink, win)
    # sinks plus recent window, causality first
    assert V(10, 0, 4, 3) and V(10, 3, 4, 3) and not V(10, 4, 4, 3)
    assert V(10, 8, 4, 3) and not V(10, 7, 4, 3) and V(10, 10, 4, 3)
    assert not V(2, 3, 4, 3)          # sink never overrides causality
    assert V(100, 50, 0, 51) and not V(100, 49, 0, 51)
    # the window start clamps at 0
    assert all(V(5, j, 0, 100) for j in range(6))


def test_tile_map_closed_form(oracle_mod):
    """The brute-force tile map equals the closed form
    j0 <= p1 and (win <= 0 or j0 < min(sink, p1+1) or j0+bk-1 >= max(0, p0-win+1)),
    the query-block generalisation of fc_attn_tile_in_window ("attention.cu")."""
    for n in (1, 7, 16, 33, 70):
        for bq, bk in ((1, 1), (4, 4), (16, 8), (8, 16), (128, 128)):
            for sink, win in ((0, 0), (0, 1), (4, 0), (4, 1), (4, 16), (2, 5), (0, 70), (9, 3)):
                m = oracle_mod.tile_map(n, bq, bk, sink, win)
                for qt in range(m.shape[0]):
                    p0, p1 = qt * bq, min(n, qt * bq + bq) - 1
                    for kt in range(m.shape[1]):
                        j0 = kt * bk
                        want = j0 <= p1 and (win <= 0 or j0 < min(sink, p1 + 1)
                                             or j0 + bk - 1 >= max(0, p0 - win + 1))
                        assert bool(m[qt, kt]) == want, (n, bq, bk, sink, win, qt, kt)


def test_shadow_read_rule(oracle_mod):
    """Q4_0 readers ("attention.cu", 4-bit KV cache section): sink rows always
    come from the fp16 sink copy; with a shadow window the last shadow_win
    positions before the query come from the fp16 ring, but only while the ring
    (256 rows, lapping at 256) still holds them; everything else is Q4_0."""
    R = oracle_mod.reads_fp16
    L = 1000
    # sinks
    assert R(999, 0, L, 4, 0) and R(999, 3, L, 4, 0) and not R(999, 4, L, 4, 0)
    # no window: only sinks
    assert not any(R(999, s, L, 0, 0) for s in range(1000))
    # window of 64 for the last query: keys 936..999
    assert not R(999, 935, L, 0, 64) and R(999, 936, L, 0, 64) and R(999, 999, L, 0, 64)
    # window of 256, query 999: keys > 743 and ring holds rows >= 744
    assert R(999, 744, L, 0, 256) and not R(999, 743, L, 0, 256)
    # earlier query of a batch: its window reaches rows the ring has lapped
    assert not R(600, 599, L, 0, 256)      # row 599 < 744 was overwritten by row 855
    assert R(900, 899, L, 0, 256)


# ------------------------------------------------------------ attention

def dense_reference(q, k, v, sink, win, kv_sel=None):
    """Independent formulation: dense masked score matrix + scipy softmax.

    kv_sel, when given, is (kbody, vbody, kf16, vf16, use_f16[p, s]) picking the
    key copy per (query, key) with a precomputed boolean matrix."""
    n, Hq, hd = q.shape
    L = k.shape[0] if kv_sel is None else kv_sel[0].shape[0]
    Hkv = k.shape[1] if kv_sel is None else kv_sel[0].shape[1]
    G = Hq // Hkv
    P = np.arange(n)[:, None]
    J = np.arange(L)[None, :]
    mask = J <= P
    if win > 0:
        mask &= (J < sink) | (J >= P - win + 1)
    out = np.zeros((n, Hq, hd))
    for h in range(Hq):
        g = h // G
        qh = q[:, h, :].astype(np.float64)
        if kv_sel is None:
            kh = k[:, g, :].astype(np.float64)
            vh = v[:, g, :].astype(np.float64)
            S = qh @ kh.T / math.sqrt(hd)
            S = np.where(mask, S, -np.inf)
            out[:, h, :] = softmax(S, axis=1) @ vh
        else:
            kb, vb, kf, vf, use = kv_sel
            Sb = qh @ kb[:, g, :].T / math.sqrt(hd)
            Sf = qh @ kf[:, g, :].T / math.sqrt(hd)
            S = np.where(use, Sf, Sb)
            S = np.where(mask, S, -np.inf)
            Pm = softmax(S, axis=1)
            out[:, h, :] = (Pm * ~use) @ vb[:, g, :] + (Pm * use) @ vf[:, g, :]
    return out


CASES = [(0, 0), (0, 1), (4, 0), (4, 1), (4, 16), (0, 40), (9, 3), (2, 5), (3, 7)]


@pytest.mark.parametrize("sink,win", CASES)
def test_brute_force_f32(oracle_mod, sink, win):
    from workloads import prefill_inputs
    q, k, v = prefill_inputs(37, 6, 2, 32, seed=100 + sink * 7 + win)
    got = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=sink, win=win)
    want = dense_reference(q, k, v, sink, win)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shadow", [(0, 0), (4, 0), (4, 256), (8, 256), (2, 16)])
def test_brute_force_q4(oracle_mod, shadow):
    """Q4_0 cache: keys read per the shadow rule; the dense reference gets the
    copies from numpy's fp16 cast and the Q4_0 decode, and the rule as a mask."""
    from workloads import prefill_inputs
    n = 300
    q, k, v = prefill_inputs(n, 4, 2, 64, seed=55)
    ss, sw = shadow
    got = oracle_mod.prefill(q, k, v, kv_fmt="q4_0", sink=0, win=0, shadow_sink=ss,
                             shadow_win=sw)
    kb = oracle_mod.q4_decode(oracle_mod.q4_encode(k), 64)
    vb = oracle_mod.q4_decode(oracle_mod.q4_encode(v), 64)
    kf = k.astype(np.float16).astype(np.float64)
    vf = v.astype(np.float16).astype(np.float64)
    P = np.arange(n)[:, None]
    S = np.arange(n)[None, :]
    use = (S < ss) | ((sw > 0) & (S > P - sw) & (S >= n - 256))
    want = dense_reference(q, None, None, 0, 0, kv_sel=(kb, vb, kf, vf, use))
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


def test_window_extremes_equal_full(oracle_mod):
    from workloads import prefill_inputs
    n = 50
    q, k, v = prefill_inputs(n, 4, 1, 32, seed=9)
    full = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
    for sink, win in ((0, -3), (5, 0), (0, n), (3, n + 10), (0, 10**6)):
        got = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=sink, win=win)
        assert np.array_equal(got, full), (sink, win)


def test_row0_returns_v0_and_win1_returns_vp(oracle_mod):
    from workloads import prefill_inputs
    q, k, v = prefill_inputs(40, 8, 2, 64, seed=21)
    out = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
    for h in range(8):
        assert np.array_equal(out[0, h], v[0, h // 4].astype(np.float64))
    out1 = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=1)
    for p in range(40):
        for h in range(8):
            assert np.array_equal(out1[p, h], v[p, h // 4].astype(np.float64))


def test_win1_q4_reads_the_right_copy(oracle_mod):
    """With only the query's own key visible, the output is that key's V as the
    cache stores it for this reader: fp16 for sink or live ring rows, else Q4_0."""
    from workloads import prefill_inputs
    n = 400
    q, k, v = prefill_inputs(n, 2, 1, 64, seed=77)
    out = oracle_mod.prefill(q, k, v, kv_fmt="q4_0", sink=0, win=1, shadow_sink=3,
                             shadow_win=256)
    vq = oracle_mod.q4_decode(oracle_mod.q4_encode(v), 64)
    vf = v.astype(np.float16).astype(np.float64)
    for p in range(n):
        want = vf[p, 0] if (p < 3 or p >= n - 256) else vq[p, 0]
        assert np.array_equal(out[p, 0], want), p
    assert not np.array_equal(vf[10, 0], vq[10, 0])


def test_identical_keys_give_mean_of_visible_v(oracle_mod):
    rng = np.random.default_rng(4)
    n, hd = 30, 32
    q = rng.standard_normal((n, 2, hd)).astype(np.float32)
    k = np.repeat(rng.standard_normal((1, 1, hd)).astype(np.float32), n, axis=0)
    v = rng.standard_normal((n, 1, hd)).astype(np.float32)
    for sink, win in ((0, 0), (2, 4), (0, 3)):
        out = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=sink, win=win)
        for p in range(n):
            vis = [j for j in range(p + 1)
                   if win <= 0 or j < sink or j >= p - win + 1]
            want = v[vis, 0].astype(np.float64).mean(axis=0)
            np.testing.assert_allclose(out[p, 0], want, rtol=1e-13, atol=1e-14)
            np.testing.assert_allclose(out[p, 1], want, rtol=1e-13, atol=1e-14)


def test_gqa_equals_mha_with_replicated_kv(oracle_mod):
    from workloads import prefill_inputs
    q, k, v = prefill_inputs(33, 8, 2, 32, seed=31)
    for fmt in ("f32", "q4_0"):
        gqa = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=2, win=9, shadow_sink=2,
                                 shadow_win=256 if fmt == "q4_0" else 0)
        k_rep = np.repeat(k, 4, axis=1)
        v_rep = np.repeat(v, 4, axis=1)
        mha = oracle_mod.prefill(q, k_rep, v_rep, kv_fmt=fmt, sink=2, win=9, shadow_sink=2,
                                 shadow_win=256 if fmt == "q4_0" else 0)
        assert np.array_equal(gqa, mha)


def test_decode_equals_prefill_row(oracle_mod):
    from workloads import prefill_inputs
    n = 90
    q, k, v = prefill_inputs(n, 4, 2, 64, seed=8)
    for fmt, ss, sw in (("f32", 0, 0), ("q4_0", 4, 0), ("q4_0", 4, 256)):
        full = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=4, win=20, shadow_sink=ss,
                                  shadow_win=sw)
        p = n - 1
        dec = oracle_mod.decode(q[p], p, k, v, kv_fmt=fmt, sink=4, win=20, shadow_sink=ss,
                                shadow_win=sw)
        np.testing.assert_array_equal(dec, full[p])


# ------------------------------------------------- split-KV decode + merge

def test_dec_plan():
    from oracle import oracle as o
    # about 256 keys per split, split length a multiple of 16, capped
    assert o.dec_plan(32768, 256, 128) == (128, 256)
    assert o.dec_plan(1, 256, 128) == (1, 16)
    assert o.dec_plan(300, 256, 128) == (2, 160)
    assert o.dec_plan(32768, 256, 16) == (16, 2048)
    assert o.dec_plan(1000, 100, 4) == (4, 256)
    for L in range(1, 3000, 37):
        for kps, cap in ((256, 128), (64, 7), (16, 1000)):
            ns, sl = o.dec_plan(L, kps, cap)
            assert sl % 16 == 0 and 1 <= ns <= cap
            assert (ns - 1) * sl < L <= ns * sl


@pytest.mark.parametrize("fmt,sink,win", [("f32", 0, 0), ("f32", 4, 100), ("q4_0", 4, 0),
                                          ("q4_0", 0, 33)])
def test_split_invariance(oracle_mod, fmt, sink, win):
    """Merging the partials of any split plan reproduces the unsplit softmax
    (to fp64 rounding), empty splits included."""
    from workloads import decode_slot_inputs
    L = 700
    q, k, v = decode_slot_inputs(L, 4, 2, 64, seed=12, slot=0)
    p = L - 1
    kk = oracle_mod.KVValues(k, fmt)
    vv = oracle_mod.KVValues(v, fmt)
    ref = oracle_mod.attention(q[None], np.array([p], np.int32), kk, vv, sink=sink, win=win,
                               shadow_sink=4 if fmt == "q4_0" else 0)[0]
    for kps, cap in ((256, 128), (16, 1000), (100, 3), (1000, 1)):
        ns, sl = oracle_mod.dec_plan(L, kps, cap)
        parts = [oracle_mod.partial(q, p, s * sl, min(L, (s + 1) * sl), kk, vv, sink=sink,
                                    win=win, shadow_sink=4 if fmt == "q4_0" else 0)
                 for s in range(ns)]
        # plus explicit empty partials past the plan
        parts.append((np.full(4, -np.inf), np.zeros(4), np.zeros((4, 64))))
        for h in range(4):
            m = np.array([pp[0][h] for pp in parts])
            l = np.array([pp[1][h] for pp in parts])
            acc = np.array([pp[2][h] for pp in parts])
            got = oracle_mod.combine(m, l, acc)
            np.testing.assert_allclose(got, ref[h], rtol=1e-12, atol=1e-12)


def test_partial_empty_range(oracle_mod):
    from workloads import decode_slot_inputs
    q, k, v = decode_slot_inputs(100, 2, 1, 32, seed=1, slot=3)
    kk = oracle_mod.KVValues(k, "f32")
    vv = oracle_mod.KVValues(v, "f32")
    m, l, acc = oracle_mod.partial(q, 99, 20, 60, kk, vv, sink=4, win=10)
    assert np.all(m == -np.inf) and np.all(l == 0) and np.all(acc == 0)


def test_combine_closed_form(oracle_mod):
    """Two partials with hand-picked numbers: M = 2, weights e^-1 and 1."""
    m = np.array([1.0, 2.0])
    l = np.array([3.0, 5.0])
    acc = np.array([[6.0, 0.0], [0.0, 10.0]])
    w = math.exp(-1.0)
    want = np.array([6.0 * w, 10.0]) / (3.0 * w + 5.0)
    np.testing.assert_allclose(oracle_mod.combine(m, l, acc), want, rtol=1e-15)
    with pytest.raises(ValueError):
        oracle_mod.combine(np.array([-np.inf]), np.array([0.0]), np.zeros((1, 2)))


# ------------------------------------------- log-sum-exp and state merging

def test_lse_of_a_single_key(oracle_mod):
    """Causal row 0 sees key 0 only: its lse is that one score, scale q.k0."""
    from workloads import prefill_inputs
    q, k, v = prefill_inputs(5, 4, 2, 32, seed=41)
    _, lse = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0, with_lse=True)
    for h in range(4):
        want = (1.0 / math.sqrt(32)) * float(np.dot(q[0, h].astype(np.float64),
                                                    k[0, h // 2].astype(np.float64)))
        assert lse[0, h] == pytest.approx(want, rel=1e-13, abs=1e-13)


def test_lse_of_equal_scores_counts_the_visible_keys(oracle_mod):
    """With every key row equal, all visible scores are one value s, so
    lse = s + log |S(p)|, which counts the attended set."""
    from workloads import prefill_inputs
    n, hd = 60, 32
    q, k, v = prefill_inputs(n, 2, 1, hd, seed=42)
    k[:] = k[7]
    for sink, win in ((0, 0), (3, 10), (0, 1)):
        _, lse = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=sink, win=win, with_lse=True)
        for p in (0, 1, 9, 30, n - 1):
            count = sum(oracle_mod.visible(p, j, sink, win) for j in range(p + 1))
            for h in range(2):
                s = (1.0 / math.sqrt(hd)) * float(np.dot(q[p, h].astype(np.float64),
                                                         k[0, 0].astype(np.float64)))
                assert lse[p, h] == pytest.approx(s + math.log(count), rel=1e-12, abs=1e-12)


def test_merge_of_disjoint_states_is_the_union(oracle_mod):
    """Attention over keys [0, c) and over [c, p] (each normalised, with its
    lse) merge into attention over [0, p] and its lse."""
    from workloads import decode_slot_inputs
    L, H, D = 300, 4, 64
    q, k, v = decode_slot_inputs(L, H, 2, D, seed=43, slot=1)
    p = L - 1
    kk, vv = oracle_mod.KVValues(k, "f32"), oracle_mod.KVValues(v, "f32")
    full, full_lse = oracle_mod.attention(q[None], np.array([p], np.int32), kk, vv, sink=0,
                                          win=0, with_lse=True)
    for c in (1, 17, 150, 299):
        states = []
        for lo, hi in ((0, c), (c, L)):
            m, l, acc = oracle_mod.partial(q, p, lo, hi, kk, vv, sink=0, win=0)
            states.append((acc / l[:, None], m + np.log(l)))
        (po, pl), (so, sl) = states
        out, lse = oracle_mod.merge_attn_states(po[None], pl[:, None], so[None], sl[:, None])
        np.testing.assert_allclose(out[0], full[0], rtol=2e-6, atol=2e-6)
        np.testing.assert_allclose(lse[:, 0], full_lse[0], rtol=1e-6, atol=1e-6)


def test_merge_edge_cases_stated_by_the_pages(oracle_mod):
    """"vt/ops.h" MergeAttnStates: +inf lse counts as -inf; both -inf gives
    the prefix output and -inf; tokens from with_context on take the suffix."""
    T, H, D = 4, 2, 8
    rng = np.random.default_rng(5)
    po = rng.standard_normal((T, H, D)).astype(np.float32)
    so = rng.standard_normal((T, H, D)).astype(np.float32)
    pl = np.array([[np.inf, -np.inf, 0.5, -np.inf], [1.0, 2.0, np.inf, 0.0]], np.float32)
    sl = np.array([[0.25, -np.inf, 0.5, 3.0], [1.0, np.inf, np.inf, -np.inf]], np.float32)
    out, lse = oracle_mod.merge_attn_states(po, pl, so, sl)
    # token 0, head 0: prefix +inf -> -inf, so the suffix alone
    np.testing.assert_array_equal(out[0, 0], so[0, 0])
    assert lse[0, 0] == np.float32(0.25)
    # token 1, head 0: both -inf -> prefix output, lse -inf
    np.testing.assert_array_equal(out[1, 0], po[1, 0])
    assert lse[0, 1] == -np.inf
    # token 2, head 0: equal lses -> the mean, lse + log 2
    np.testing.assert_allclose(out[2, 0], (po[2, 0].astype(np.float64) + so[2, 0]) / 2,
                               rtol=1e-15)
    assert lse[0, 2] == pytest.approx(0.5 + math.log(2.0), rel=1e-15)
    # token 3, head 0: prefix -inf -> the suffix alone
    np.testing.assert_array_equal(out[3, 0], so[3, 0])
    # token 0, head 1: equal finite lses
    np.testing.assert_allclose(out[0, 1], (po[0, 1].astype(np.float64) + so[0, 1]) / 2,
                               rtol=1e-15)
    # token 1, head 1: suffix +inf -> -inf, the prefix alone, its lse
    np.testing.assert_array_equal(out[1, 1], po[1, 1])
    assert lse[1, 1] == np.float32(2.0)
    # token 2, head 1: both +inf -> both -inf -> prefix output, -inf
    np.testing.assert_array_equal(out[2, 1], po[2, 1])
    assert lse[1, 2] == -np.inf
    # token 3, head 1: weights 1 and e^-inf = 0 -> the prefix
    np.testing.assert_array_equal(out[3, 1], po[3, 1])
    assert lse[1, 3] == 0.0
    # tokens from with_context = 2 on take the suffix output and lse verbatim
    out2, lse2 = oracle_mod.merge_attn_states(po, pl, so, sl, with_context=2)
    np.testing.assert_array_equal(out2[2:], so[2:])
    np.testing.assert_array_equal(lse2[:, 2:], sl[:, 2:])
    np.testing.assert_array_equal(out2[:2], out[:2])


# ------------------------------------------- chunked prefill (pos0 > 0)

def test_tile_map_closed_form_with_offset_queries(oracle_mod):
    """A chunk of n queries at positions pos0.. over keys 0..pos0+n-1: the
    brute-force map equals the closed form on absolute positions
    p0 = pos0 + qt*bq, p1 = pos0 + min(n, qt*bq+bq) - 1, with key tiles up to
    pos0 + n; pos0 = 0 is the map of a plain prefill."""
    for pos0 in (0, 1, 5, 16, 40):
        for n in (1, 7, 33):
            for bq, bk in ((4, 4), (16, 8), (8, 16)):
                for sink, win in ((0, 0), (4, 1), (4, 16), (0, 70), (9, 3)):
                    m = oracle_mod.tile_map(n, bq, bk, sink, win, pos0=pos0)
                    assert m.shape == (-(-n // bq), -(-(pos0 + n) // bk))
                    for qt in range(m.shape[0]):
                        p0 = pos0 + qt * bq
                        p1 = pos0 + min(n, qt * bq + bq) - 1
                        for kt in range(m.shape[1]):
                            j0 = kt * bk
                            want = j0 <= p1 and (win <= 0 or j0 < min(sink, p1 + 1)
                                                 or j0 + bk - 1 >= max(0, p0 - win + 1))
                            assert bool(m[qt, kt]) == want, (pos0, n, bq, bk, sink, win, qt, kt)


@pytest.mark.parametrize("fmt,shadow", [("f32", (0, 0)), ("q4_0", (4, 0)), ("q4_0", (4, 256))])
def test_chunk_equals_rows_of_the_whole_prefill(oracle_mod, fmt, shadow):
    """Queries pos0.. of a chunk over the cache rows 0..pos0+n-1 are the rows
    pos0.. of the prefill of all pos0+n tokens, lse included: a row's attention
    depends on its position and the cache only."""
    from workloads import prefill_inputs
    L = 300
    q, k, v = prefill_inputs(L, 4, 2, 64, seed=61)
    whole, whole_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=3, win=50,
                                          shadow_sink=shadow[0], shadow_win=shadow[1],
                                          with_lse=True)
    for pos0 in (1, 37, 128, 299):
        part, part_lse = oracle_mod.prefill(q[pos0:], k, v, kv_fmt=fmt, sink=3, win=50,
                                            shadow_sink=shadow[0], shadow_win=shadow[1],
                                            with_lse=True, pos0=pos0)
        np.testing.assert_array_equal(part, whole[pos0:])
        np.testing.assert_array_equal(part_lse, whole_lse[pos0:])


# ------------------------------------------------ fp16 and fp8 KV formats

def test_e4m3_golden(oracle_mod):
    for name, xb, cb in golden_lines("e4m3.txt"):
        x = f32_from_hex(xb)
        assert oracle_mod.e4m3(x) == int(cb, 16), name


def test_e4m3_codes_round_trip(oracle_mod):
    """Every finite code decodes to a value that encodes back to it, the values
    are strictly increasing over the positive codes and span [2^-9, 448]."""
    vals = []
    for c in range(256):
        v = oracle_mod.e4m3_value(c)
        if c in (0x7f, 0xff):
            assert math.isnan(v)
            continue
        assert oracle_mod.e4m3(v) == c, hex(c)
        if c <= 0x7e:
            vals.append(v)
    assert vals == sorted(vals) and len(set(vals)) == len(vals)
    assert vals[1] == 2.0 ** -9 and vals[-1] == 448.0


def test_e4m3_is_nearest_even_with_saturation(oracle_mod):
    """Against the table of all finite values: the encoding of x is the value
    nearest to x, ties to the even code, and +-448 beyond."""
    table = np.array([oracle_mod.e4m3_value(c) for c in range(0x7f)])  # 0 .. 448
    rng = np.random.default_rng(3)
    xs = np.concatenate([rng.standard_normal(3000) * 30, rng.standard_normal(500) * 0.01,
                         (table[:-1] + table[1:]) / 2, table, [500.0, 463.9, 464.0]])
    for x in xs.astype(np.float32):
        c = oracle_mod.e4m3(float(x))
        a = abs(float(x))
        if a >= 448.0:
            assert c & 0x7f == 0x7e
            continue
        d = np.abs(table - a)
        best = np.flatnonzero(d == d.min())
        want = best[0] if len(best) == 1 else [b for b in best if b % 2 == 0][0]
        assert c & 0x7f == want, (x, hex(c))
        assert (c >> 7) == (1 if np.signbit(x) else 0)


def test_fp8_kv_store_and_read_use_the_scale(oracle_mod):
    """Store x / scale, read byte * scale: with scale s the reader sees
    s * e4m3(x / s); a power-of-two scale only moves the grid."""
    rng = np.random.default_rng(8)
    x = (rng.standard_normal(2000) * 3).astype(np.float32)
    for s in (1.0, 0.25, 8.0, 0.0123):
        q = oracle_mod.e4m3_store(x, s)
        got = oracle_mod.e4m3_load(q, s)
        for i in range(0, 2000, 97):
            t = np.float32(x[i] / np.float32(s))
            assert q[i] == oracle_mod.e4m3(t)
            assert got[i] == float(np.float32(np.float32(oracle_mod.e4m3_value(q[i])) * np.float32(s)))
    q1 = oracle_mod.e4m3_store(x * 4, 4.0)
    assert np.array_equal(q1, oracle_mod.e4m3_store(x, 1.0))


def test_f16_and_fp8_caches_are_attention_over_their_values(oracle_mod):
    """An f16 (fp8) cache is attention over the fp16 rounding (the fp8 store
    and read) of the same rows: equal to an fp32 cache holding those values."""
    from workloads import prefill_inputs
    q, k, v = prefill_inputs(64, 4, 2, 32, seed=17)
    k16 = oracle_mod.f16_to_f64(oracle_mod.f16_rne(k)).astype(np.float32)
    v16 = oracle_mod.f16_to_f64(oracle_mod.f16_rne(v)).astype(np.float32)
    a = oracle_mod.prefill(q, k, v, kv_fmt="f16", sink=2, win=9)
    b = oracle_mod.prefill(q, k16, v16, kv_fmt="f32", sink=2, win=9)
    np.testing.assert_array_equal(a, b)
    k8 = oracle_mod.e4m3_load(oracle_mod.e4m3_store(k, 0.5), 0.5).astype(np.float32)
    v8 = oracle_mod.e4m3_load(oracle_mod.e4m3_store(v, 2.0), 2.0).astype(np.float32)
    a = oracle_mod.prefill(q, k, v, kv_fmt="fp8_e4m3", sink=0, win=0, k_scale=0.5, v_scale=2.0)
    b = oracle_mod.prefill(q, k8, v8, kv_fmt="f32", sink=0, win=0)
    np.testing.assert_array_equal(a, b)
