"""Checkpoint and resume of a KV cache.

The planes' bytes are the whole state of a cache: their layout is a defined
interface that the host may read and write ("attention.cu", "4-bit KV cache
(Q4_0 blocks)"; "vt/ops.h", the paged fp8 KV cache). So a save is a byte copy
of the planes to the host (here through a file) and a resume a byte copy into
fresh device memory, with no fa_kv_init. Appending and decoding on after a
resume must give planes and outputs bit-identical to the uninterrupted cache,
and outputs within tolerance of the oracle."""
import numpy as np
import pytest
import torch

from gpu_util import (POISON_BYTE, assert_close, build_cache, check_guards, fa, fmt_code,
                      guarded, run_decode)
from workloads import decode_slot_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fmt,shadow_sink,shadow_win,sink,win", [
    ("q4_0", 4, 256, 4, 160),
    ("fp8_e4m3", 0, 0, 4, 0),
    ("f16", 0, 0, 0, 0),
    ("f32", 0, 0, 2, 100),
])
def test_checkpoint_resume_is_a_byte_copy(oracle_mod, tmp_path, fmt, shadow_sink, shadow_win,
                                          sink, win):
    m = fa()
    nslots, hq, hkv, hd, max_seq = 2, 8, 2, 128, 640
    L1, L2 = 300, 420  # the Q4_0 ring of 256 rows has wrapped at both lengths
    ks, vs = (0.5, 2.0) if fmt == "fp8_e4m3" else (1.0, 1.0)
    slots = [decode_slot_inputs(L2, hq, hkv, hd, seed=61, slot=s) for s in range(nslots)]
    q = np.stack([s[0] for s in slots])
    K = np.stack([s[1] for s in slots])
    V = np.stack([s[2] for s in slots])
    kp, vp, _ = build_cache(K[:, :L1], V[:, :L1], kv_fmt=fmt, shadow_sink=shadow_sink,
                            shadow_win=shadow_win, max_seq=max_seq, k_scale=ks, v_scale=vs)

    # save: the planes' bytes to a file; resume: the bytes into fresh memory
    path = tmp_path / "kv_cache.npz"
    np.savez(path, k=kp.cpu().numpy(), v=vp.cpu().numpy())
    saved = np.load(path)
    kr = guarded(kp.numel(), torch.uint8, fill_byte=POISON_BYTE)
    vr = guarded(vp.numel(), torch.uint8, fill_byte=POISON_BYTE)
    kr.copy_(torch.from_numpy(saved["k"]))
    vr.copy_(torch.from_numpy(saved["v"]))

    # both caches go on: append rows L1 .. L2-1, decode at position L2-1
    k_new = torch.from_numpy(np.ascontiguousarray(K[:, L1:L2])).cuda()
    v_new = torch.from_numpy(np.ascontiguousarray(V[:, L1:L2])).cuda()
    pos0 = torch.full((nslots,), L1, dtype=torch.int32, device="cuda")
    for kpl, vpl in ((kp, vp), (kr, vr)):
        m.kv_append(k_new, v_new, kpl, vpl, pos0, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq,
                    kv_fmt=fmt_code(fmt), shadow_sink=shadow_sink, shadow_win=shadow_win)
    assert m.get_device_error() == m.OK
    check_guards(("resumed k planes", kr), ("resumed v planes", vr))
    assert torch.equal(kp, kr) and torch.equal(vp, vr)

    pos = [L2 - 1] * nslots
    kw = dict(hkv=hkv, hd=hd, max_seq=max_seq, sink=sink, win=win, kv_fmt=fmt,
              shadow_sink=shadow_sink, shadow_win=shadow_win)
    out_a = run_decode(q, kp, vp, pos, **kw)
    out_b = run_decode(q, kr, vr, pos, **kw)
    assert np.array_equal(out_a, out_b)
    for s in range(nslots):
        want = oracle_mod.decode(q[s], L2 - 1, K[s], V[s], kv_fmt=fmt, sink=sink, win=win,
                                 shadow_sink=shadow_sink, shadow_win=shadow_win, k_scale=ks,
                                 v_scale=vs)
        assert_close(out_b[s], want, f"{fmt} slot {s} after resume")
