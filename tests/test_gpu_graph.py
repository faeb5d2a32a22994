"""The decode step captured once in a CUDA graph and replayed.

fa_kv_append, fa_decode and fa_decode_combine read the slots' positions from
device memory, so one capture of [append the new row, decode, combine,
advance the positions] serves every later step: the host only refreshes the
inputs of the static buffers before each replay. Each replay's output must
match the oracle's decode at that step's positions, like an eager call."""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, fa, fmt_code
from workloads import decode_slot_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv_fmt,shadow", [("q4_0", (4, 256)), ("f32", (0, 0)), ("f16", (0, 0)),
                                           ("fp8_e4m3", (0, 0))])
def test_decode_step_graph_replay(oracle_mod, kv_fmt, shadow):
    nslots, hq, hkv, hd, max_seq = 3, 16, 2, 128, 1024
    sink, win, kps = 4, 0, 64
    ss, sw = shadow
    lens0 = [100, 300, 517]  # rows cached before the first step
    steps = 4
    Lmax = max(lens0) + steps
    q_all, k_all, v_all = [], [], []
    for u in range(nslots):
        # one query per step: draw them from a second stream of the slot's seed
        _, ku, vu = decode_slot_inputs(Lmax, hq, hkv, hd, seed=777, slot=u)
        qs = [decode_slot_inputs(1, hq, hkv, hd, seed=9000 + 31 * step, slot=u)[0]
              for step in range(steps)]
        q_all.append(np.stack(qs))
        k_all.append(ku)
        v_all.append(vu)
    m = fa()
    code = fmt_code(kv_fmt)
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    for u, L in enumerate(lens0):
        m.kv_append(torch.from_numpy(k_all[u][None, :L]).cuda(),
                    torch.from_numpy(v_all[u][None, :L]).cuda(),
                    kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code, shadow_sink=ss, shadow_win=sw)
    max_splits = -(-max_seq // kps)
    ws = torch.empty(m.decode_workspace_bytes(nslots, hq, hd, max_splits), dtype=torch.uint8,
                     device="cuda")
    q_s = torch.zeros(nslots, hq, hd, dtype=torch.float32, device="cuda")
    k_s = torch.zeros(nslots, 1, hkv, hd, dtype=torch.float32, device="cuda")
    v_s = torch.zeros_like(k_s)
    out = torch.zeros(nslots, hq, hd, dtype=torch.float32, device="cuda")
    pos = torch.tensor(lens0, dtype=torch.int32, device="cuda")  # the new row's position
    common = dict(n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code, shadow_sink=ss,
                  shadow_win=sw)

    def step():
        m.kv_append(k_s, v_s, kp, vp, pos, **common)
        m.decode(q_s, kp, vp, pos, n_q_heads=hq, sink=sink, win=win, split_keys=kps,
                 max_splits=max_splits, workspace=ws, **common)
        m.decode_combine(ws, out, nslots=nslots, n_q_heads=hq, head_dim=hd,
                         max_splits=max_splits)
        pos.add_(1)

    # one-time set-up inside the library (kernel attributes) happens on the
    # first calls: make them outside the capture, on a copy of the positions
    # that the warm-up decode reads but nothing appends to
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        pos_w = pos - 1  # the last cached row of every slot
        m.decode(q_s, kp, vp, pos_w, n_q_heads=hq, sink=sink, win=win, split_keys=kps,
                 max_splits=max_splits, workspace=ws, **common)
        m.decode_combine(ws, out, nslots=nslots, n_q_heads=hq, head_dim=hd,
                         max_splits=max_splits)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()

    for t in range(steps):
        p = [L + t for L in lens0]
        q_s.copy_(torch.from_numpy(np.stack([q_all[u][t] for u in range(nslots)])))
        k_s.copy_(torch.from_numpy(np.stack([k_all[u][p[u]][None] for u in range(nslots)])))
        v_s.copy_(torch.from_numpy(np.stack([v_all[u][p[u]][None] for u in range(nslots)])))
        graph.replay()
        torch.cuda.synchronize()
        st = m.get_device_error()
        assert st == m.OK, m.status_string(st)
        got = out.cpu().numpy()
        for u in range(nslots):
            want = oracle_mod.decode(q_all[u][t], p[u], k_all[u], v_all[u], kv_fmt=kv_fmt,
                                     sink=sink, win=win, shadow_sink=ss, shadow_win=sw)
            assert_close(got[u], want, f"{kv_fmt} step {t} slot {u}")
    assert pos.cpu().tolist() == [L + steps for L in lens0]


def test_kernel_events_eager_and_in_a_captured_graph():
    """fa_set_kernel_events brackets the split-decode kernel: a plain call
    records the events, and a call captured in a CUDA graph records them on
    every replay."""
    m = fa()
    nslots, hq, hkv, hd, max_seq = 2, 16, 2, 128, 512
    code = fmt_code("f16")
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    k = torch.randn(nslots, 300, hkv, hd, device="cuda")
    m.kv_append(k, k, kp, vp, torch.zeros(nslots, dtype=torch.int32, device="cuda"),
                n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code)
    q = torch.randn(nslots, hq, hd, device="cuda")
    pos = torch.full((nslots,), 299, dtype=torch.int32, device="cuda")
    max_splits = 2
    ws = torch.empty(m.decode_workspace_bytes(nslots, hq, hd, max_splits), dtype=torch.uint8,
                     device="cuda")
    kw = dict(n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, sink=0, win=0,
              kv_fmt=code, split_keys=256, max_splits=max_splits, workspace=ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for e in (e0, e1, g0, g1):  # create the CUDA events
        e.record()
    torch.cuda.synchronize()
    try:
        m.set_kernel_events(e0, e1)
        m.decode(q, kp, vp, pos, **kw)
        torch.cuda.synchronize()
        assert e0.elapsed_time(e1) > 0.0
        m.set_kernel_events(g0, g1)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.decode(q, kp, vp, pos, **kw)
        m.set_kernel_events(None, None)
        for _ in range(2):
            graph.replay()
            torch.cuda.synchronize()
            assert g0.elapsed_time(g1) > 0.0
    finally:
        m.set_kernel_events(None, None)
    assert m.get_device_error() == m.OK
