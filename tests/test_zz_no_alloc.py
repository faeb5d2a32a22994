"""fa_decode_noalloc: decode for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc (a plugin whose host owns all device
memory, or a serving loop where allocation is banned because it can
synchronise the device). fa_decode_noalloc keeps its partials in the
library's fixed device array instead of a caller workspace. This file checks,
through the C ABI, that two calls in a row give what the existing
fa_decode + fa_decode_combine give, and that problems too large for the
fixed array are rejected. It is collected last and needs nothing from the
other test files."""
import numpy as np
import pytest
import torch

from gpu_util import MAX_ABS, REL_L2, errors, fa

pytestmark = pytest.mark.gpu


def _cache(m, rng, nslots, hkv, hd, max_seq, lens, shadow_sink):
    kp = m.alloc_planes(nslots, m.KV_Q4_0, hkv, max_seq, hd)
    vp = m.alloc_planes(nslots, m.KV_Q4_0, hkv, max_seq, hd)
    pb = m.kv_plane_bytes(m.KV_Q4_0, hkv, max_seq, hd)
    for u, L in enumerate(lens):
        k = torch.from_numpy(rng.standard_normal((1, L, hkv, hd)).astype(np.float32)).cuda()
        v = torch.from_numpy(rng.standard_normal((1, L, hkv, hd)).astype(np.float32)).cuda()
        m.kv_append(k, v, kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=m.KV_Q4_0, shadow_sink=shadow_sink)
    return kp, vp


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


def test_noalloc_matches_decode_twice_in_a_row():
    m = fa()
    rng = np.random.default_rng(31337)
    nslots, hq, hkv, hd, max_seq = 4, 16, 2, 256, 4096
    lens = [4096, 1500, 2900, 700]
    kp, vp = _cache(m, rng, nslots, hkv, hd, max_seq, lens, shadow_sink=4)
    kw = dict(n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, sink=4, win=0,
              kv_fmt=m.KV_Q4_0, shadow_sink=4, shadow_win=0, split_keys=256, max_splits=16)
    for call, pos_list in enumerate(([L - 1 for L in lens], [1000, 1499, 64, 699])):
        q = torch.from_numpy(rng.standard_normal((nslots, hq, hd)).astype(np.float32)).cuda()
        pos = torch.tensor(pos_list, dtype=torch.int32, device="cuda")
        want = _with_workspace(m, q, kp, vp, pos, **kw)
        out = torch.full((nslots, hq, hd), float("nan"), device="cuda")
        m.decode_noalloc(q, kp, vp, pos, out, **kw)
        assert m.get_device_error() == m.OK
        got = out.cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}"
        ma, rl = errors(got, want)
        assert ma <= MAX_ABS and rl <= REL_L2, f"call {call}: max_abs={ma:.3e} rel_l2={rl:.3e}"


def test_noalloc_rejects_oversized_problems():
    m = fa()
    L = m.lib()
    # 256 slots x 16 heads x 256 dims needs more than the fixed 8 MiB of partials
    st = L.fa_decode_noalloc(256, 256, 256, 256, 256, 16, 1, 256, 32768, 0, 0, m.KV_Q4_0, 0,
                             0, 256, 128, 256, None)
    assert st == m.ERR_WORKSPACE
    assert m.get_device_error() == m.OK
