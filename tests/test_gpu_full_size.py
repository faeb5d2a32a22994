"""Every output of the full-size workloads against the oracle, through the C ABI.

The workloads are the ones the benchmark times, at their full sizes and
launched as the benchmark launches them: the 8192-token prefills over fp32,
Q4_0 (fp16 shadows of 4 sinks and the 256 newest rows), fp16 and fp8 caches,
full causal and with 4 sinks + a 1024-key window; the chunked prefill of
tokens 4096..8191 over 8192 cache rows; and the 32-slot x 32768-key decodes
over Q4_0, fp16 and fp8 caches. Nothing is sampled: every query row of every
head (its output, and the log-sum-exp of the fa_prefill_lse variant) and
every slot of every decode is compared, within max-abs 5e-3 and relative L2
2e-3 for outputs and max-abs 5e-3 for log-sum-exps (the tolerances of every
other parity test); the prefills' visited-tile maps are compared bit for bit.

The measured errors are appended to the file named by FA_PARITY_LOG when it
is set."""
import numpy as np
import pytest
import torch

from gpu_util import (assert_close, errors, fa, fmt_code, record_parity, run_chunk, run_decode,
                      run_prefill)
from workloads import BY_NAME, WORKLOADS, decode_slot_inputs, prefill_inputs

pytestmark = pytest.mark.gpu

LSE_ATOL = 5e-3

PREFILLS = [w.name for w in WORKLOADS if w.kind == "prefill"]
DECODES = [w.name for w in WORKLOADS if w.kind == "decode"]


def _lse_err(got, want_t):
    assert np.all(np.isfinite(got)), "non-finite lse"
    return float(np.max(np.abs(got - want_t)))


@pytest.mark.parametrize("name", PREFILLS)
def test_prefill_every_row(oracle_mod, name):
    """fa_prefill (the benchmark's kernel) and fa_prefill_lse, all n x Hq rows."""
    w = BY_NAME[name]
    q, k, v = prefill_inputs(w.n, w.n_q_heads, w.n_kv_heads, w.head_dim, w.seed)
    kw = dict(kv_fmt=w.kv_fmt, sink=w.sink, win=w.win, shadow_sink=w.shadow_sink,
              shadow_win=w.shadow_win, k_scale=w.k_scale, v_scale=w.v_scale)
    got, tm = run_prefill(q, k, v, tile_map=True, **kw)
    got_l, lse = run_prefill(q, k, v, lse=True, **kw)
    want, want_lse = oracle_mod.prefill(q, k, v, with_lse=True, **kw)
    ma, rl = assert_close(got, want, name)
    ma_l, rl_l = assert_close(got_l, want, name + " (lse variant)")
    le = _lse_err(lse, want_lse.T)
    assert le <= LSE_ATOL, f"{name}: lse max-abs {le:.3g}"
    bq, bk = fa().prefill_tile_shape(w.head_dim)
    assert np.array_equal(tm, oracle_mod.tile_map(w.n, bq, bk, w.sink, w.win))
    record_parity(name, rows=int(w.n * w.n_q_heads), max_abs=ma, rel_l2=rl,
                  lse_variant_max_abs=ma_l, lse_variant_rel_l2=rl_l, lse_max_abs=le)


def test_prefill_chunk_every_row(oracle_mod):
    """The benchmark's chunk: queries at 4096..8191 over cache rows 0..8191
    of the 8192-token fp32 workload (fa_prefill_chunk with lse and tile map)."""
    w = BY_NAME["prefill_f32_n8192_h16x2_d256"]
    q, k, v = prefill_inputs(w.n, w.n_q_heads, w.n_kv_heads, w.head_dim, w.seed)
    pos0 = w.n // 2
    out, lse, tm = run_chunk(q[pos0:], k, v, pos0, hq=w.n_q_heads, hkv=w.n_kv_heads,
                             hd=w.head_dim, sink=w.sink, win=w.win, kv_fmt=w.kv_fmt,
                             shadow=(0, 0), want_map=True)
    want, want_lse = oracle_mod.prefill(q[pos0:], k, v, kv_fmt=w.kv_fmt, sink=w.sink, win=w.win,
                                        with_lse=True, pos0=pos0)
    ma, rl = assert_close(out, want, "chunk")
    le = _lse_err(lse, want_lse.T)
    assert le <= LSE_ATOL, f"chunk: lse max-abs {le:.3g}"
    bq, bk = fa().prefill_tile_shape(w.head_dim)
    assert np.array_equal(tm, oracle_mod.tile_map(w.n - pos0, bq, bk, w.sink, w.win, pos0=pos0))
    record_parity("prefill_chunk_f32_pos4096_n4096_h16x2_d256", rows=int((w.n - pos0) * 16),
                  max_abs=ma, rel_l2=rl, lse_max_abs=le)


@pytest.mark.parametrize("name", DECODES)
def test_decode_every_slot(oracle_mod, name):
    """All 32 slots of the 32 x 32768 decode, with the benchmark's split plan
    (256-key splits, 128 at most). The oracle's answer for each slot is taken
    as the slot is drawn, so no more than one slot's keys are held on the host."""
    w = BY_NAME[name]
    m = fa()
    code = fmt_code(w.kv_fmt)
    L = w.n
    kp = m.alloc_planes(w.nslots, code, w.n_kv_heads, L, w.head_dim, scale=w.k_scale)
    vp = m.alloc_planes(w.nslots, code, w.n_kv_heads, L, w.head_dim, scale=w.v_scale)
    pb = m.kv_plane_bytes(code, w.n_kv_heads, L, w.head_dim)
    qs, wants = [], []
    for u in range(w.nslots):
        qu, ku, vu = decode_slot_inputs(L, w.n_q_heads, w.n_kv_heads, w.head_dim, w.seed, u)
        qs.append(qu)
        m.kv_append(torch.from_numpy(ku[None]).cuda(), torch.from_numpy(vu[None]).cuda(),
                    kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"),
                    n_kv_heads=w.n_kv_heads, head_dim=w.head_dim, max_seq=L, kv_fmt=code,
                    shadow_sink=w.shadow_sink, shadow_win=w.shadow_win)
        wants.append(oracle_mod.decode(qu, L - 1, ku, vu, kv_fmt=w.kv_fmt, sink=w.sink,
                                       win=w.win, shadow_sink=w.shadow_sink,
                                       shadow_win=w.shadow_win, k_scale=w.k_scale,
                                       v_scale=w.v_scale))
        del ku, vu
    got = run_decode(np.stack(qs), kp, vp, np.full(w.nslots, L - 1, np.int32),
                     hkv=w.n_kv_heads, hd=w.head_dim, max_seq=L, sink=w.sink, win=w.win,
                     kv_fmt=w.kv_fmt, shadow_sink=w.shadow_sink, shadow_win=w.shadow_win,
                     split_keys=w.split_keys, max_splits=-(-L // w.split_keys))
    want = np.stack(wants)
    worst = 0.0
    for u in range(w.nslots):
        ma_u, _ = assert_close(got[u], want[u], f"{name} slot {u}")
        worst = max(worst, ma_u)
    ma, rl = errors(got, want)
    record_parity(name, slots=w.nslots, max_abs=ma, rel_l2=rl, worst_slot_max_abs=worst)
