"""Parity of the fp16 and fp8 e4m3fn KV cache formats with the CPU oracle,
through the C ABI.

Stored bytes are compared bit for bit: binary16 rounded to nearest even
("qwen38_batched.rs", the BQ_KV16 half-width cache), and e4m3fn of x / scale
rounded to nearest even with saturation to +-448 ("vt/ops.h",
ReshapeAndCacheFp8 and the e4m3fn format). Attention outputs (prefill, chunked
prefill, decode) use the tolerance of every other format, max-abs 5e-3 and
relative L2 2e-3: the oracle attends over exactly the values a reader of the
cache sees (float(byte) * scale for fp8), and the kernels add only the fp16
rounding of their MMA operands."""

import numpy as np
import pytest
import torch

from gpu_util import assert_close, build_cache, fa, fmt_code, run_decode, run_prefill
from workloads import decode_slot_inputs, prefill_inputs

pytestmark = pytest.mark.gpu


def body_bytes(planes, u, code, hkv, max_seq, hd, L):
    """Rows 0..L-1 of slot u's plane body as [L][hkv][row_bytes] uint8."""
    m = fa()
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    row, body, _, _ = m.kv_plane_layout(code, hkv, max_seq, hd)
    raw = planes[u * pb + body:u * pb + body + hkv * max_seq * row].cpu().numpy()
    return raw.reshape(hkv, max_seq, row)[:, :L].transpose(1, 0, 2)


@pytest.mark.parametrize("hd", [64, 128, 256])
def test_append_f16_bitexact(oracle_mod, hd):
    m = fa()
    nslots, n, hkv, max_seq = 2, 37, 2, 100
    rng = np.random.default_rng(hd)
    k = (rng.standard_normal((nslots, n, hkv, hd)) * 3).astype(np.float32)
    v = (rng.standard_normal((nslots, n, hkv, hd)) * 3).astype(np.float32)
    k[0, 0, 0, :6] = [65504.0, 65520.0, 1e-8, -2.0 ** -25, 6.1e-5, -0.0]  # edges of binary16
    code = fmt_code("f16")
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd)
    pos0 = torch.tensor([0, 41], dtype=torch.int32, device="cuda")
    m.kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kp, vp, pos0,
                n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code)
    assert m.get_device_error() == m.OK
    for u, p0 in enumerate((0, 41)):
        for planes, x in ((kp, k), (vp, v)):
            got = body_bytes(planes, u, code, hkv, max_seq, hd, p0 + n)[p0:]
            want = oracle_mod.f16_rne(x[u])
            assert np.array_equal(got.view(np.uint16), want), (hd, u)


FP8_EDGES = np.array([0.0, -0.0, 1.0, 1.0625, 1.1875, 448.0, 449.0, 464.0, 480.0, 1e6, -1e6,
                      2.0 ** -6, 2.0 ** -9, 2.0 ** -10, 3 * 2.0 ** -10, 7.5 * 2.0 ** -9, 240.0,
                      0.1, -2.0, -7 * 2.0 ** -9, 2.0 ** -12], np.float32)


@pytest.mark.parametrize("hd,k_scale,v_scale", [(64, 1.0, 1.0), (128, 0.37, 4.0),
                                                (256, 0.0123, 2.5)])
def test_append_fp8_bitexact(oracle_mod, hd, k_scale, v_scale):
    m = fa()
    nslots, n, hkv, max_seq = 2, 45, 2, 64
    rng = np.random.default_rng(hd + 1)
    k = (rng.standard_normal((nslots, n, hkv, hd)) * 3).astype(np.float32)
    v = (rng.standard_normal((nslots, n, hkv, hd)) * 3).astype(np.float32)
    # values that land on the format's ties, subnormals and saturation
    k[1, 3, 1, :len(FP8_EDGES)] = FP8_EDGES * np.float32(k_scale)
    v[0, 7, 0, :len(FP8_EDGES)] = FP8_EDGES * np.float32(v_scale)
    code = fmt_code("fp8_e4m3")
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=k_scale)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=v_scale)
    pos0 = torch.tensor([19, 0], dtype=torch.int32, device="cuda")
    m.kv_append(torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda(), kp, vp, pos0,
                n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code)
    assert m.get_device_error() == m.OK
    so = m.kv_scale_offset(code, hkv, max_seq, hd)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    for u, p0 in enumerate((19, 0)):
        for planes, x, c in ((kp, k, k_scale), (vp, v, v_scale)):
            got = body_bytes(planes, u, code, hkv, max_seq, hd, p0 + n)[p0:]
            assert np.array_equal(got, oracle_mod.e4m3_store(x[u], c)), (hd, u, c)
            sc = planes[u * pb + so:u * pb + so + 4].cpu().numpy().view(np.float32)[0]
            assert sc == np.float32(c)


def test_append_fp8_infinities_saturate(oracle_mod):
    """+-inf take the saturating conversion to +-448 (0x7e, 0xfe), the
    oracle's reading of saturation to finite."""
    m = fa()
    hkv, hd, max_seq = 1, 64, 4
    x = np.zeros((1, 1, hkv, hd), np.float32)
    x[0, 0, 0, :4] = [np.inf, -np.inf, 500.0, -500.0]
    code = fmt_code("fp8_e4m3")
    kp = m.alloc_planes(1, code, hkv, max_seq, hd)
    vp = m.alloc_planes(1, code, hkv, max_seq, hd)
    m.kv_append(torch.from_numpy(x).cuda(), torch.from_numpy(x).cuda(), kp, vp,
                torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv, head_dim=hd,
                max_seq=max_seq, kv_fmt=code)
    assert m.get_device_error() == m.OK
    got = body_bytes(kp, 0, code, hkv, max_seq, hd, 1)[0, 0, :4]
    want = oracle_mod.e4m3_store(x[0, 0, 0, :4], 1.0)
    assert got.tolist() == want.tolist() == [0x7e, 0xfe, 0x7e, 0xfe]


def test_fp8_plane_without_scale_is_not_written():
    """A plane whose scale slot holds 0 (never set) rejects the append on the
    device: FA_ERR_DEVICE, and the body stays as it was."""
    m = fa()
    hkv, hd, max_seq = 2, 64, 16
    code = fmt_code("fp8_e4m3")
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    kp = torch.zeros(pb, dtype=torch.uint8, device="cuda")
    vp = torch.zeros(pb, dtype=torch.uint8, device="cuda")
    x = torch.ones(1, 3, hkv, hd, device="cuda")
    m.kv_append(x, x, kp, vp, torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                head_dim=hd, max_seq=max_seq, kv_fmt=code)
    assert m.get_device_error() == m.ERR_DEVICE
    assert int(kp.count_nonzero()) == 0 and int(vp.count_nonzero()) == 0
    with pytest.raises(m.FAError):
        m.kv_set_scale(kp, code, hkv, max_seq, hd, 0.0)


PREFILL_CASES = [
    # n, hq, hkv, hd, sink, win, fmt, k_scale, v_scale, spare rows of the planes
    (1, 8, 2, 64, 0, 0, "f16", 1.0, 1.0, 0),
    (129, 4, 2, 128, 9, 3, "f16", 1.0, 1.0, 27),
    (300, 16, 2, 256, 4, 100, "f16", 1.0, 1.0, 300),
    (700, 16, 2, 256, 0, 0, "f16", 1.0, 1.0, 5),
    (1, 8, 2, 64, 0, 0, "fp8_e4m3", 1.0, 1.0, 0),
    (200, 8, 1, 64, 0, 0, "fp8_e4m3", 0.5, 2.0, 56),
    (333, 16, 2, 256, 2, 40, "fp8_e4m3", 0.37, 1.3, 0),
    (520, 16, 2, 256, 0, 0, "fp8_e4m3", 1.0, 1.0, 100),
]


@pytest.mark.parametrize("case", PREFILL_CASES, ids=lambda c: "-".join(map(str, c)))
def test_prefill_formats(oracle_mod, case):
    n, hq, hkv, hd, sink, win, fmt, ks, vs, spare = case
    q, k, v = prefill_inputs(n, hq, hkv, hd, seed=4000 + n + hd)
    got = run_prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, max_seq=n + spare, k_scale=ks,
                      v_scale=vs)
    want = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, k_scale=ks, v_scale=vs)
    assert_close(got, want, str(case))


@pytest.mark.parametrize("fmt,ks,vs", [("f16", 1.0, 1.0), ("fp8_e4m3", 0.6, 1.7)])
def test_prefill_chunk_formats(oracle_mod, fmt, ks, vs):
    """Queries at positions 517..816 over cache rows 0..816 of planes with
    room for 1000 rows, the context appended in a first call."""
    m = fa()
    pos0, n, hq, hkv, hd, sink, win, max_seq = 517, 300, 16, 2, 256, 4, 200, 1000
    q_all, k, v = prefill_inputs(pos0 + n, hq, hkv, hd, seed=4321)
    q = q_all[pos0:]
    code = fmt_code(fmt)
    kp = m.alloc_planes(1, code, hkv, max_seq, hd, scale=ks)
    vp = m.alloc_planes(1, code, hkv, max_seq, hd, scale=vs)
    for lo, hi in ((0, pos0), (pos0, pos0 + n)):
        m.kv_append(torch.from_numpy(np.ascontiguousarray(k[None, lo:hi])).cuda(),
                    torch.from_numpy(np.ascontiguousarray(v[None, lo:hi])).cuda(), kp, vp,
                    torch.tensor([lo], dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code)
    ws = torch.empty(m.prefill_chunk_workspace_bytes(pos0, n, hq, hkv, hd), dtype=torch.uint8,
                     device="cuda")
    out = torch.full((n, hq, hd), float("nan"), dtype=torch.float32, device="cuda")
    lse = torch.full((hq, n), float("nan"), dtype=torch.float32, device="cuda")
    m.prefill_chunk(torch.from_numpy(np.ascontiguousarray(q)).cuda(), kp, vp, out, pos0, n, hq,
                    hkv, hd, sink, win, code, max_seq=max_seq, workspace=ws, lse=lse)
    st = m.get_device_error()
    assert st == m.OK, m.status_string(st)
    want, want_lse = oracle_mod.prefill(q, k, v, kv_fmt=fmt, sink=sink, win=win, pos0=pos0,
                                        with_lse=True, k_scale=ks, v_scale=vs)
    assert_close(out.cpu().numpy(), want, fmt)
    assert np.max(np.abs(lse.cpu().numpy() - want_lse.T)) <= 5e-3


DECODE_CASES = [
    # lens per slot, hq, hkv, hd, sink, win, fmt, k_scale, v_scale, split_keys, max_seq
    # (group <= 8 and fp8 head_dim >= 128 run the streaming kernel, the rest the
    # generic one)
    ((1, 17, 300, 1000), 16, 2, 256, 4, 0, "f16", 1.0, 1.0, 256, 1024),
    ((700, 64, 1500), 8, 2, 128, 4, 100, "f16", 1.0, 1.0, 64, 1600),
    ((999, 5), 16, 1, 64, 0, 0, "f16", 1.0, 1.0, 100, 1000),
    ((1, 17, 300, 1000), 16, 2, 256, 4, 0, "fp8_e4m3", 1.0, 1.0, 256, 1024),
    ((513, 2000), 8, 2, 128, 0, 0, "fp8_e4m3", 0.25, 3.0, 256, 2048),
    ((640, 640, 33), 4, 4, 64, 2, 37, "fp8_e4m3", 0.9, 0.45, 128, 700),
    # streaming kernel: groups 1, 2, 4, 8; positions 0 and tile edges; windows
    # that leave one tile, sinks past the position; a workspace of 2 entries
    ((1, 16, 17, 32, 33, 250), 2, 2, 64, 0, 0, "f16", 1.0, 1.0, 16, 256),
    ((4000, 1, 2500), 4, 1, 128, 3, 1, "f16", 1.0, 1.0, 4000, 4096),
    ((3000, 3001, 15, 2999), 8, 8, 128, 40, 16, "fp8_e4m3", 1.7, 0.3, 128, 3072),
    ((777,) * 9, 32, 4, 256, 0, 0, "fp8_e4m3", 0.5, 0.5, 256, 800),
    ((2048, 100), 16, 16, 256, 2000, 64, "f16", 1.0, 1.0, 256, 2048),
    # group 16 over fp8 (the generic kernel)
    ((1, 17, 300, 1000), 16, 1, 256, 4, 0, "fp8_e4m3", 0.5, 2.0, 256, 1024),
    ((2048, 100), 32, 2, 128, 2000, 64, "fp8_e4m3", 1.0, 1.0, 256, 2048),
    ((700, 64, 1500), 16, 1, 64, 4, 100, "fp8_e4m3", 1.3, 0.7, 64, 1600),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "-".join(map(str, c[1:])))
def test_decode_formats(oracle_mod, case):
    lens, hq, hkv, hd, sink, win, fmt, ks, vs, kps, max_seq = case
    nslots = len(lens)
    Lmax = max(lens)
    qs, kk, vv = [], [], []
    for u in range(nslots):
        qu, ku, vu = decode_slot_inputs(Lmax, hq, hkv, hd, seed=5150, slot=u)
        qs.append(qu)
        kk.append(ku)
        vv.append(vu)
    q = np.stack(qs)
    m = fa()
    code = fmt_code(fmt)
    kp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=ks)
    vp = m.alloc_planes(nslots, code, hkv, max_seq, hd, scale=vs)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    for u, L in enumerate(lens):
        m.kv_append(torch.from_numpy(kk[u][None, :L]).cuda(), torch.from_numpy(vv[u][None, :L]).cuda(),
                    kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code)
    got = run_decode(q, kp, vp, np.array(lens, np.int32) - 1, hkv=hkv, hd=hd, max_seq=max_seq,
                     sink=sink, win=win, kv_fmt=fmt, split_keys=kps)
    for u, L in enumerate(lens):
        want = oracle_mod.decode(q[u], L - 1, kk[u], vv[u], kv_fmt=fmt, sink=sink, win=win,
                                 k_scale=ks, v_scale=vs)
        assert_close(got[u], want, f"{case} slot {u}")


def test_decode_dense_noalloc_and_bad_position(oracle_mod):
    """The streaming kernel through fa_decode_noalloc (fewer entries: the
    library's fixed array) matches the oracle; a slot whose position is past
    max_seq flags FA_ERR_DEVICE and leaves the other slots right."""
    m = fa()
    lens, hq, hkv, hd, max_seq = (3000, 700, 1), 16, 2, 256, 3072
    qs, kk, vv = [], [], []
    for u in range(len(lens)):
        qu, ku, vu = decode_slot_inputs(max(lens), hq, hkv, hd, seed=6060, slot=u)
        qs.append(qu)
        kk.append(ku)
        vv.append(vu)
    q = torch.from_numpy(np.stack(qs)).cuda()
    for fmt, ks, vs in (("f16", 1.0, 1.0), ("fp8_e4m3", 0.8, 1.25)):
        code = fmt_code(fmt)
        kp = m.alloc_planes(len(lens), code, hkv, max_seq, hd, scale=ks)
        vp = m.alloc_planes(len(lens), code, hkv, max_seq, hd, scale=vs)
        pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
        for u, L in enumerate(lens):
            m.kv_append(torch.from_numpy(kk[u][None, :L]).cuda(),
                        torch.from_numpy(vv[u][None, :L]).cuda(), kp[u * pb:(u + 1) * pb],
                        vp[u * pb:(u + 1) * pb], torch.zeros(1, dtype=torch.int32, device="cuda"),
                        n_kv_heads=hkv, head_dim=hd, max_seq=max_seq, kv_fmt=code)
        out = torch.full((len(lens), hq, hd), float("nan"), device="cuda")
        pos = torch.tensor([L - 1 for L in lens], dtype=torch.int32, device="cuda")
        m.decode_noalloc(q, kp, vp, pos, out, n_q_heads=hq, n_kv_heads=hkv, head_dim=hd,
                         max_seq=max_seq, sink=4, win=0, kv_fmt=code, split_keys=256,
                         max_splits=12)
        assert m.get_device_error() == m.OK
        got = out.cpu().numpy()
        for u, L in enumerate(lens):
            want = oracle_mod.decode(qs[u], L - 1, kk[u], vv[u], kv_fmt=fmt, sink=4, win=0,
                                     k_scale=ks, v_scale=vs)
            assert_close(got[u], want, f"noalloc {fmt} slot {u}")
        bad = torch.tensor([lens[0] - 1, max_seq, lens[2] - 1], dtype=torch.int32, device="cuda")
        ws = torch.empty(m.decode_workspace_bytes(len(lens), hq, hd, 12), dtype=torch.uint8,
                         device="cuda")
        m.decode(q, kp, vp, bad, n_q_heads=hq, n_kv_heads=hkv, head_dim=hd, max_seq=max_seq,
                 sink=4, win=0, kv_fmt=code, split_keys=256, max_splits=12, workspace=ws)
        assert m.get_device_error() == m.ERR_DEVICE


@pytest.mark.parametrize("fmt", ["f32", "q4_0", "f16", "fp8_e4m3"])
def test_kv_init_zeroes_planes_and_sets_the_fp8_scale(fmt):
    m = fa()
    code = fmt_code(fmt)
    hkv, max_seq, hd, nslots = 2, 40, 64, 3
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    planes = torch.full((nslots * pb,), 0xAB, dtype=torch.uint8, device="cuda")
    m.kv_init(planes, code, hkv, max_seq, hd)
    torch.cuda.synchronize()
    host = planes.cpu().numpy().reshape(nslots, pb)
    so = m.kv_scale_offset(code, hkv, max_seq, hd)
    for u in range(nslots):
        if fmt == "fp8_e4m3":
            assert host[u, so:so + 4].view(np.float32)[0] == 1.0
            host[u, so:so + 4] = 0
        assert not host[u].any(), (fmt, u)


@pytest.mark.parametrize("fmt", ["f16", "fp8_e4m3"])
def test_decode_dense_with_two_entries(oracle_mod, fmt):
    """max_splits = 1 leaves the streaming kernel two entries per head: every
    (slot, kv head) must then be covered by at most two pieces of the
    warps' runs, whatever the slot lengths."""
    lens, hq, hkv, hd, max_seq = (2000, 17, 1, 1999), 8, 2, 128, 2048
    qs, kk, vv = [], [], []
    for u in range(len(lens)):
        qu, ku, vu = decode_slot_inputs(max(lens), hq, hkv, hd, seed=7070, slot=u)
        qs.append(qu)
        kk.append(ku)
        vv.append(vu)
    m = fa()
    code = fmt_code(fmt)
    kp = m.alloc_planes(len(lens), code, hkv, max_seq, hd)
    vp = m.alloc_planes(len(lens), code, hkv, max_seq, hd)
    pb = m.kv_plane_bytes(code, hkv, max_seq, hd)
    for u, L in enumerate(lens):
        m.kv_append(torch.from_numpy(kk[u][None, :L]).cuda(), torch.from_numpy(vv[u][None, :L]).cuda(),
                    kp[u * pb:(u + 1) * pb], vp[u * pb:(u + 1) * pb],
                    torch.zeros(1, dtype=torch.int32, device="cuda"), n_kv_heads=hkv,
                    head_dim=hd, max_seq=max_seq, kv_fmt=code)
    got = run_decode(np.stack(qs), kp, vp, np.array(lens, np.int32) - 1, hkv=hkv, hd=hd,
                     max_seq=max_seq, sink=0, win=0, kv_fmt=fmt, split_keys=4096, max_splits=1)
    for u, L in enumerate(lens):
        want = oracle_mod.decode(qs[u], L - 1, kk[u], vv[u], kv_fmt=fmt, sink=0, win=0)
        assert_close(got[u], want, f"{fmt} slot {u}")
