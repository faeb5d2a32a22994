"""fa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a plugin whose host owns all device
memory, or a serving loop where allocation is banned because it can
synchronise the device). fa_decode_noalloc keeps its partials in the
library's fixed device array instead of a caller workspace. This file checks,
through the C ABI, that two calls in a row give what the existing
fa_decode + fa_decode_combine give and what the oracle gives, over Q4_0,
fp16 (with more partials than the fixed array holds, so the call uses fewer)
and fp32 caches, and that problems too large for the fixed array are
rejected. It is collected last and needs nothing from the other test files."""
import numpy as np
import pytest
import torch

from gpu_util import MAX_ABS, REL_L2, assert_close, errors, fa

pytestmark = pytest.mark.gpu


def _cache(m, rng, code, nslots, hkv, hd, max_seq, lens, shadow_sink):
    """Planes holding rows 0..len-1 of each slot; returns them and the host K, V."""
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    ks, vs = [], []
    for u, L in enumerate(lens):
        k = rng.standard_normal((L, hkv, hd)).astype(np.float32)
        v = rng.standard_normal((L, hkv, hd)).astype(np.float32)
        m.kv_append(torch.from_numpy(k[None]).cuda(), torch.from_numpy(v[None]).cuda(),
                    kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code, shadow_sink=shadow_sink)
        ks.append(k)
        vs.append(v)
    return kp, vp, ks, vs


def _with_workspace(m, q, kp, vp, pos, **kw):
    nslots, hq, hd = q.shape
    ws = torch.empty(m.decode_workspace_bytes(nslots, hq, hd, kw["max_splits"]),
                     dtype=torch.uint8, device="cuda")
    out = torch.full((nslots, hq, hd), float("nan"), device="cuda")
    m.decode(q, kp, vp, pos, workspace=ws, **kw)
    m.decode_combine(ws, out, nslots=nslots, n_q_heads=hq, head_dim=hd,
                     max_splits=kw["max_splits"])
    assert m.get_device_error() == m.OK
    return out.cpu().numpy()


FMT_NAMES = {0: "f32", 1: "q4_0", 2: "f16"}

CASES = [
    # kv_fmt code, nslots, hq, hkv, hd, max_seq, lens, sink, shadow_sink, max_splits
    (1, 4, 16, 2, 256, 4096, [4096, 1500, 2900, 700], 4, 4, 16),
    # 32 x 16 heads x 65 entries of 256 dims need 34 MB of partials: the
    # streaming kernel is given the 15 entries that fit the fixed array
    (2, 32, 16, 2, 256, 2048, [2048 - 37 * u for u in range(32)], 4, 0, 64),
    # fp32 cache, group 4 (the generic kernel)
    (0, 3, 8, 2, 128, 1500, [1500, 333, 1], 0, 0, 8),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"{FMT_NAMES[c[0]]}-{c[1]}slots")
def test_noalloc_matches_decode_and_oracle_twice_in_a_row(oracle_mod, case):
    code, nslots, hq, hkv, hd, max_seq, lens, sink, ss, max_splits = case
    m = fa()
    rng = np.random.default_rng(31337 + code)
    kp, vp, ks, vs = _cache(m, rng, code, nslots, hkv, hd, max_seq, lens, ss)
    kw = dict(n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, sink=sink, win=0,
              kv_fmt=code, shadow_sink=ss, shadow_win=0, split_keys=256, max_splits=max_splits)
    later = [max(0, (L - 1) * 2 // 3) for L in lens]
    for call, pos_list in enumerate(([L - 1 for L in lens], later)):
        qh = rng.standard_normal((nslots, hq, hd)).astype(np.float32)
        q = torch.from_numpy(qh).cuda()
        pos = torch.tensor(pos_list, dtype=torch.int32, device="cuda")
        want = _with_workspace(m, q, kp, vp, pos, **kw)
        out = torch.full((nslots, hq, hd), float("nan"), device="cuda")
        m.decode_noalloc(q, kp, vp, pos, out, **kw)
        assert m.get_device_error() == m.OK
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}"
        ma, rl = errors(got, want)
        assert ma <= MAX_ABS and rl <= REL_L2, f"call {call}: max_abs={ma:.3e} rel_l2={rl:.3e}"
        for u, p in enumerate(pos_list):
            ref = oracle_mod.decode(qh[u], p, ks[u], vs[u], kv_fmt=FMT_NAMES[code], sink=sink,
                                    win=0, shadow_sink=ss, shadow_win=0)
            assert_close(got[u], ref, f"call {call} slot {u}")


def test_noalloc_rejects_oversized_problems():
    m = fa()
    L = m.lib()
    # 256 slots x 16 heads x 256 dims needs more than the fixed 8 MiB of partials
    st = L.fa_decode_noalloc(256, 256, 256, 256, 256, 16, 1, 256, 32768, 0, 0, m.KV_Q4_0, 0,
                             0, 256, 128, 256, None)
    assert st == m.ERR_WORKSPACE
    assert m.get_device_error() == m.OK
