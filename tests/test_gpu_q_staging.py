"""Parity of prefills large enough that the kernel stages part of Q itself.

The staging launch before the prefill kernel converts only the query tiles of
the kernel's first wave of units (one unit per SM, rounded up to whole query
tiles; two waves when the heaviest unit is short); two warps of every prefill
block convert the rest while the tensor cores run and flag each tile, and the
producer that loads a unit's Q tile waits for its flag. These cases have more
units than those first waves, on
every path that stages Q: fp32, Q4_0 (staged K/V, and the two-part prefill of
a narrow fp16 window), fp8, fp16 planes read in place, a chunk continuing a
cache, and the log-sum-exp output. The workspace starts poisoned, so flags
that were not cleared would let a producer load a tile before it is staged.
Outputs are compared with the fp64 oracle at the usual tolerance (max-abs
5e-3, relative L2 2e-3), log-sum-exps within 5e-3."""

import numpy as np
import pytest

from gpu_util import assert_close, fa, run_chunk, run_prefill
from workloads import prefill_inputs

pytestmark = pytest.mark.gpu

SEED = 7301


def _staged_in_kernel(oracle_mod, n, hq, sink, win, pos0=0):
    """Units whose Q the kernel converts itself: those past the first wave of
    units (one block per SM), or past the first two when the heaviest query
    tile visits fewer than 24 key tiles, rounded up to whole query tiles."""
    import torch

    sms = torch.cuda.get_device_properties(0).multi_processor_count
    nqt = -(-n // 128)
    units = nqt * hq
    heavy = int(oracle_mod.tile_map(n, 128, 128, sink, win, pos0=pos0)[-1].sum())
    waves = 2 if heavy < 24 else 1
    first = min(units, -(-(waves * min(units, sms)) // hq) * hq)
    return units - first


# (n, hq, hkv, hd, sink, win, fmt, (shadow_sink, shadow_win), k_scale)
CASES = [
    (3200, 16, 2, 64, 0, 0, "f32", (0, 0), 1.0),
    (3200, 32, 4, 128, 4, 300, "f32", (0, 0), 1.0),
    (1500, 32, 4, 128, 4, 300, "f32", (0, 0), 1.0),
    (1400, 32, 4, 128, 0, 0, "q4_0", (4, 256), 1.0),
    (1400, 32, 4, 128, 0, 0, "q4_0", (4, 64), 1.0),
    (1400, 32, 4, 128, 0, 0, "f16", (0, 0), 1.0),
    (1400, 32, 4, 128, 0, 0, "fp8_e4m3", (0, 0), 4.0),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_kernel_stages_q(oracle_mod, case):
    n, hq, hkv, hd, sink, win, fmt, (ss, sw), ksc = case
    assert _staged_in_kernel(oracle_mod, n, hq, sink, win) > 0, "must reach past the first waves"
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=SEED + n + hd)
    got, got_lse = run_prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss,
                               shadow_win=sw, k_scale=ksc, lse=True)
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, shadow_sink=ss,
                                        shadow_win=sw, k_scale=ksc, with_lse=True)
    assert_close(got, want, str(case))
    err = np.max(np.abs(got_lse - want_lse.T))
    assert np.all(np.isfinite(got_lse)) and err <= 5e-3, f"{case}: lse max-abs {err:.3g}"


def test_prefill_chunk_kernel_stages_q(oracle_mod):
    """Queries 700..2099 over 2100 cached rows, 32 q heads."""
    pos0, n, hq, hkv, hd, sink, win = 700, 1400, 32, 4, 128, 4, 1024
    assert _staged_in_kernel(oracle_mod, n, hq, sink, win, pos0) > 0
    q_all, k, v = prefill_inputs(pos0 + n, hq, hkv, hd, seed=SEED + 1)
    q = q_all[pos0:]
    out, lse, _ = run_chunk(q, k, v, pos0, hq=hq, hkv=hkv, hd=hd, sink=sink, win=win,
                            kv_fmt="f32", shadow=(0, 0))
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=sink, win=win,
                                        with_lse=True, pos0=pos0)
    assert_close(out, want, "chunk")
    err = np.max(np.abs(lse - want_lse.T))
    assert np.all(np.isfinite(lse)) and err <= 5e-3, f"chunk: lse max-abs {err:.3g}"


def test_prefill_repeat_same_workspace(oracle_mod):
    """Two prefills in a row on one workspace: the second must not see the
    first one's flags (each call clears them before its kernel runs)."""
    import torch

    from gpu_util import build_cache, fmt_code

    m = fa()
    n, hq, hkv, hd = 3200, 16, 2, 64
    assert _staged_in_kernel(oracle_mod, n, hq, 0, 0) > 0
    q1, k, v = prefill_inputs(n, hq, hkv, hd, seed=SEED + 2)
    q2 = prefill_inputs(n, hq, hkv, hd, seed=SEED + 3)[0]
    kp, vp, max_seq = build_cache(k, v, kv_fmt="f32")
    ws = torch.empty(m.prefill_workspace_bytes(n, hq, hkv, hd), dtype=torch.uint8, device="cuda")
    outs = []
    for q in (q1, q2):
        out = torch.empty((n, hq, hd), dtype=torch.float32, device="cuda")
        m.prefill(torch.from_numpy(q).cuda(), kp, vp, out, n, hq, hkv, hd, 0, 0, fmt_code("f32"),
                  max_seq=max_seq, workspace=ws)
        outs.append(out)
    assert m.get_device_error() == m.OK
    for q, out in zip((q1, q2), outs):
        assert_close(out.cpu().numpy(), oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0),
                     "repeat")


def test_prefill_graph_replay_kernel_stages_q(oracle_mod):
    """A prefill captured once in a CUDA graph and replayed with new queries:
    each replay's staging launch clears the counters and flags again, so the
    kernel waits for this replay's Q tiles, not the last one's."""
    import torch

    from gpu_util import build_cache, fmt_code

    m = fa()
    n, hq, hkv, hd = 3200, 16, 2, 64
    assert _staged_in_kernel(oracle_mod, n, hq, 0, 0) > 0
    _, k, v = prefill_inputs(n, hq, hkv, hd, seed=SEED + 4)
    qs = [prefill_inputs(n, hq, hkv, hd, seed=SEED + 5 + i)[0] for i in range(3)]
    kp, vp, max_seq = build_cache(k, v, kv_fmt="f32")
    ws = torch.empty(m.prefill_workspace_bytes(n, hq, hkv, hd), dtype=torch.uint8, device="cuda")
    q_s = torch.zeros(n, hq, hd, dtype=torch.float32, device="cuda")
    out = torch.zeros(n, hq, hd, dtype=torch.float32, device="cuda")

    def step():
        m.prefill(q_s, kp, vp, out, n, hq, hkv, hd, 0, 0, fmt_code("f32"), max_seq=max_seq,
                  workspace=ws)

    step()  # one-time set-up inside the library, outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for i, q in enumerate(qs):
        q_s.copy_(torch.from_numpy(q))
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        st = m.get_device_error()
        assert st == m.OK, m.status_string(st)
        want = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
        assert_close(out.cpu().numpy(), want, f"replay {i}")
