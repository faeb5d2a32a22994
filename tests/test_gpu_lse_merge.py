"""Parity of the prefill's log-sum-exp output and of the attention-state merge
(through the C ABI) with the CPU oracle.

lse: the oracle's log sum_j exp(s_j) in fp64; the kernel's scores come from
fp16 operands (relative rounding 2^-11 per element) and fp32 accumulation, so
a score of a few units carries an error of order 1e-3 and so does the lse:
max-abs 5e-3, the tolerance of the outputs.
merge: fp32 arithmetic against the fp64 oracle on the same fp32 inputs; the
weights and sums lose a few ulp: relative and absolute 2e-6."""
import math

import numpy as np
import pytest
import torch

from gpu_util import assert_close, build_cache, fa, fmt_code
from workloads import prefill_inputs

pytestmark = pytest.mark.gpu

LSE_ATOL = 5e-3


def run_prefill_lse(q, k, v, *, hq, hkv, hd, sink, win, kv_fmt, shadow=(0, 0)):
    m = fa()
    n = q.shape[0]
    code = fmt_code(kv_fmt)
    kp, vp, _ = build_cache(k, v, kv_fmt=kv_fmt, shadow_sink=shadow[0], shadow_win=shadow[1],
                            max_seq=n)
    ws = torch.empty(m.prefill_workspace_bytes(n, hq, hkv, hd), dtype=torch.uint8, device="cuda")
    out = torch.full((n, hq, hd), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((hq, n), float("nan"), dtype=torch.float32, device="cuda")
    qd = torch.from_numpy(np.ascontiguousarray(q)).cuda()
    m.prefill(qd, kp, vp, out, n, hq, hkv, hd, sink, win, code, max_seq=n,
              shadow_sink=shadow[0], shadow_win=shadow[1], workspace=ws, lse=lse)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    return out.cpu().numpy(), lse.cpu().numpy()


LSE_CASES = [
    # n, hq, hkv, hd, sink, win, fmt, shadow
    (1, 8, 2, 64, 0, 0, "f32", (0, 0)),
    (129, 4, 2, 128, 9, 3, "f32", (0, 0)),
    (300, 16, 2, 256, 4, 100, "f32", (0, 0)),
    (700, 16, 2, 256, 0, 0, "f32", (0, 0)),
    (520, 16, 2, 256, 0, 0, "q4_0", (4, 256)),
    (257, 4, 1, 128, 2, 40, "q4_0", (4, 256)),
]


@pytest.mark.parametrize("case", LSE_CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_lse_small(oracle_mod, case):
    n, hq, hkv, hd, sink, win, fmt, shadow = case
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=515 + n)
    out, lse = run_prefill_lse(q, k, v, hq=hq, hkv=hkv, hd=hd, sink=sink, win=win, kv_fmt=fmt,
                               shadow=shadow)
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win,
                                        shadow_sink=shadow[0], shadow_win=shadow[1],
                                        with_lse=True)
    assert_close(out, want, str(case))
    err = np.max(np.abs(lse - want_lse.T))
    assert np.all(np.isfinite(lse)) and err <= LSE_ATOL, f"{case}: lse max-abs {err:.3g}"


def run_merge(po, pl, so, sl, with_context=-1, want_lse=True):
    m = fa()
    T, H, D = po.shape
    out = torch.full((T, H, D), float("nan"), dtype=torch.float32, device="cuda")
    out_lse = torch.full((H, T), float("nan"), dtype=torch.float32, device="cuda") \
        if want_lse else None
    t = [torch.from_numpy(np.ascontiguousarray(x)).cuda() for x in (po, pl, so, sl)]
    m.merge_attn_states(out, out_lse, *t, prefill_tokens_with_context=with_context)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (out_lse.cpu().numpy() if want_lse else None)


def merge_inputs(T, H, D, seed):
    rng = np.random.default_rng(seed)
    po = rng.standard_normal((T, H, D)).astype(np.float32)
    so = rng.standard_normal((T, H, D)).astype(np.float32)
    pl = (rng.standard_normal((H, T)) * 4).astype(np.float32)
    sl = (rng.standard_normal((H, T)) * 4).astype(np.float32)
    # the edge cases the page states, scattered over the rows
    pl[0 % H, ::7] = np.inf
    sl[1 % H, ::11] = np.inf
    pl[2 % H, ::5] = -np.inf
    sl[2 % H, ::5] = -np.inf
    sl[3 % H, ::3] = -np.inf
    return po, pl, so, sl


@pytest.mark.parametrize("T,H,D,wc", [(1, 1, 4, -1), (300, 16, 256, -1), (300, 16, 256, 120),
                                      (77, 8, 64, 0), (1000, 4, 128, 2000)])
def test_merge_attn_states(oracle_mod, T, H, D, wc):
    po, pl, so, sl = merge_inputs(T, H, D, seed=T + H + D)
    out, lse = run_merge(po, pl, so, sl, wc)
    want, want_lse = oracle_mod.merge_attn_states(po, pl, so, sl, with_context=wc)
    np.testing.assert_allclose(out, want, rtol=2e-6, atol=2e-6)
    fin = np.isfinite(want_lse)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.array_equal(lse[~fin], want_lse[~fin])
    np.testing.assert_allclose(lse[fin], want_lse[fin], rtol=2e-6, atol=2e-6)
    out2, _ = run_merge(po, pl, so, sl, wc, want_lse=False)
    assert np.array_equal(out2, out)


def test_merge_of_a_prefill_state_with_empty_and_with_itself(oracle_mod):
    """A prefill output and its lse merged with an empty state (-inf lse) is
    unchanged; merged with itself, the output is unchanged and the lse grows
    by log 2."""
    n, hq, hkv, hd = 200, 8, 2, 128
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=99)
    out, lse = run_prefill_lse(q, k, v, hq=hq, hkv=hkv, hd=hd, sink=0, win=0, kv_fmt="f32")
    empty = np.full_like(lse, -np.inf)
    got, got_lse = run_merge(out, lse, np.zeros_like(out), empty)
    assert np.array_equal(got, out) and np.array_equal(got_lse, lse)
    got, got_lse = run_merge(out, lse, out, lse)
    np.testing.assert_allclose(got, out, rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(got_lse, lse + math.log(2.0), rtol=1e-6, atol=1e-6)
