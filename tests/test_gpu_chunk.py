"""Parity of the chunked prefill (queries at positions pos0.. over the cache
rows 0..pos0+n-1) with the CPU oracle, through the C ABI.

The cache is filled as a caller continuing a sequence fills it: the context
rows 0..pos0-1 in one append, the chunk's rows pos0.. in a second. Outputs:
max-abs 5e-3 and relative L2 2e-3 (as every prefill); lse max-abs 5e-3 (the
scores' fp16 operand rounding, as for fa_prefill_lse); the visited-tile map
bit-exact."""
import numpy as np
import pytest
import torch

from gpu_util import assert_close, fa, fmt_code, run_chunk
from workloads import prefill_inputs

pytestmark = pytest.mark.gpu

CHUNK_CASES = [
    # pos0, n, hq, hkv, hd, sink, win, fmt, shadow
    (1, 1, 8, 2, 64, 0, 0, "f32", (0, 0)),
    (100, 1, 8, 2, 64, 4, 16, "f32", (0, 0)),
    (128, 128, 8, 2, 128, 0, 0, "f32", (0, 0)),
    (300, 200, 16, 2, 256, 0, 0, "f32", (0, 0)),
    (517, 300, 16, 2, 256, 4, 200, "f32", (0, 0)),
    (64, 700, 4, 1, 128, 9, 3, "f32", (0, 0)),
    (1000, 130, 16, 2, 256, 0, 0, "q4_0", (4, 256)),
    (250, 260, 8, 2, 64, 4, 1, "q4_0", (8, 256)),
    (333, 77, 4, 1, 128, 2, 40, "q4_0", (4, 0)),
    # fp16 windows narrower than the ring: which copy a query reads depends on
    # the query (the prefill runs as two merged parts)
    (0, 300, 8, 2, 128, 0, 0, "q4_0", (4, 64)),
    (0, 200, 16, 2, 256, 0, 0, "q4_0", (2, 100)),
    (517, 300, 16, 2, 256, 4, 200, "q4_0", (4, 64)),
    (1000, 130, 16, 2, 256, 0, 0, "q4_0", (8, 255)),
    (250, 260, 8, 2, 64, 4, 1, "q4_0", (0, 1)),
    (64, 700, 4, 1, 128, 9, 3, "q4_0", (4, 17)),
    (300, 1, 8, 2, 64, 0, 0, "q4_0", (4, 128)),
]


@pytest.mark.parametrize("case", CHUNK_CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_chunk(oracle_mod, case):
    pos0, n, hq, hkv, hd, sink, win, fmt, shadow = case
    L = pos0 + n
    q_all, k, v = prefill_inputs(L, hq, hkv, hd, seed=900 + pos0)
    q = q_all[pos0:]
    out, lse, tm = run_chunk(q, k, v, pos0, hq=hq, hkv=hkv, hd=hd, sink=sink, win=win,
                             kv_fmt=fmt, shadow=shadow, want_map=True)
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win,
                                        shadow_sink=shadow[0], shadow_win=shadow[1],
                                        with_lse=True, pos0=pos0)
    assert_close(out, want, str(case))
    err = np.max(np.abs(lse - want_lse.T))
    assert np.all(np.isfinite(lse)) and err <= 5e-3, f"{case}: lse max-abs {err:.3g}"
    bq, bk = fa().prefill_tile_shape(hd)
    assert np.array_equal(tm, oracle_mod.tile_map(n, bq, bk, sink, win, pos0=pos0))


@pytest.mark.parametrize("fmt,shadow", [("f32", (0, 0)), ("q4_0", (4, 256)), ("q4_0", (4, 64))])
def test_prefill_in_chunks(oracle_mod, fmt, shadow):
    """A 1000-token sequence prefilled in three chunks (300, 1, 699 tokens),
    each over the cache grown so far. With an fp32 cache the chunks are the
    rows of one prefill of all 1000 tokens; with Q4_0 and the 256-row fp16
    ring, each chunk reads the ring as it was when the chunk ran, so each is
    checked against the oracle's prefill of that chunk."""
    hq, hkv, hd, sink, win = 16, 2, 256, 4, 256
    L = 1000
    q, k, v = prefill_inputs(L, hq, hkv, hd, seed=977)
    whole = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=sink, win=win) if fmt == "f32" \
        else None
    ss, sw = shadow
    m = fa()
    code = fmt_code(fmt)
    kp = m.alloc_planes(1, code, hkv, L, hd)
    vp = m.alloc_planes(1, code, hkv, L, hd)
    got = []
    for lo, hi in ((0, 300), (300, 301), (301, 1000)):
        m.kv_append(torch.from_numpy(np.ascontiguousarray(k[None, lo:hi])).cuda(),
                    torch.from_numpy(np.ascontiguousarray(v[None, lo:hi])).cuda(), kp, vp,
                    torch.tensor([lo], dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=L, kv_fmt=code, shadow_sink=ss, shadow_win=sw)
        n = hi - lo
        ws = torch.empty(m.prefill_chunk_workspace_bytes(lo, n, hq, hkv, hd, kv_fmt=code,
                                                         shadow_win=sw),
                         dtype=torch.uint8, device="cuda")
        out = torch.full((n, hq, hd), float("nan"), dtype=torch.float32, device="cuda")
        m.prefill_chunk(torch.from_numpy(np.ascontiguousarray(q[lo:hi])).cuda(), kp, vp, out, lo,
                        n, hq, hkv, hd, sink, win, code, max_seq=L, shadow_sink=ss,
                        shadow_win=sw, workspace=ws)
        got.append(out.cpu().numpy())
        if whole is not None:
            want = whole[lo:hi]
        else:
            want = oracle_mod.prefill(q[lo:hi], k, v, kv_fmt=fmt, sink=sink, win=win,
                                      shadow_sink=ss, shadow_win=sw, pos0=lo)
        assert_close(got[-1], want, f"{fmt} chunk {lo}..{hi}")
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)


def test_prefill_chunk_rejects_positions_past_the_cache():
    m = fa()
    ws = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    x = torch.zeros(4, 8, 64, device="cuda")
    kp = m.alloc_planes(1, 0, 2, 16, 64)
    with pytest.raises(m.FAError):  # pos0 + n > max_seq
        m.prefill_chunk(x, kp, kp, x, 13, 4, 8, 2, 64, 0, 0, 0, max_seq=16, workspace=ws)
    with pytest.raises(m.FAError):
        m.prefill_chunk(x, kp, kp, x, -1, 4, 8, 2, 64, 0, 0, 0, max_seq=16, workspace=ws)
