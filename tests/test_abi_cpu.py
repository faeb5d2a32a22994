"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/fa.h declares, reports the documented plane and
workspace sizes, and rejects bad arguments before touching a device."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fa():
    from causal_gqa_flash_attn_gb300 import build
    build.build()
    import causal_gqa_flash_attn_gb300 as fa
    fa.lib()
    return fa


def header_functions():
    text = open(os.path.join(ROOT, "include", "fa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_exports_every_declared_symbol(fa):
    names = header_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(fa.lib(), name), name
    assert set(names) == set(fa.SIGNATURES)


def test_version_and_status_strings(fa):
    assert fa.version() >= 100
    for s in range(7):
        assert fa.status_string(s)
    assert "unknown" in fa.status_string(99)


def test_plane_sizes(fa):
    # Q4_0 row = hd/32 blocks of 18 bytes ("attention.cu", fc_kvq4_row_bytes)
    for hd, rb in ((64, 36), (128, 72), (256, 144)):
        row, body, sink, ring = fa.kv_plane_layout(fa.KV_Q4_0, 2, 1000, hd)
        assert row == rb and body == 0
        assert sink == ((2 * 1000 * rb + 255) // 256) * 256
        assert ring == sink + ((2 * 8 * hd * 2 + 255) // 256) * 256
        pb = fa.kv_plane_bytes(fa.KV_Q4_0, 2, 1000, hd)
        assert pb == ring + ((2 * 256 * hd * 2 + 255) // 256) * 256
        assert pb % 256 == 0
        row, body, sink, ring = fa.kv_plane_layout(fa.KV_F32, 2, 1000, hd)
        assert row == 4 * hd and sink == 0 and ring == 0
        assert fa.kv_plane_bytes(fa.KV_F32, 2, 1000, hd) == ((2 * 1000 * 4 * hd + 255) // 256) * 256
    assert fa.kv_plane_bytes(fa.KV_F32, 2, 1000, 96) == 0
    assert fa.kv_plane_bytes(7, 2, 1000, 64) == 0
    assert fa.kv_plane_bytes(fa.KV_F32, 0, 1000, 64) == 0


def test_workspace_sizes(fa):
    n, hq, hkv, hd = 8192, 16, 2, 256
    assert fa.prefill_workspace_bytes(n, hq, hkv, hd) >= 2 * (n * hq * hd + 2 * hkv * n * hd)

    def up256(x):
        return (x + 255) // 256 * 256

    # the layout fa.h documents: 256-byte header (work queues), one 4-byte Q-ready
    # flag per (query tile, q head), then fp16 Q [n][Hq][hd], K and V [Hkv][rows][hd]
    for n, hq, hkv, hd in ((8192, 16, 2, 256), (1500, 32, 4, 128), (1, 8, 1, 64)):
        units = -(-n // 128) * hq
        want = 256 + up256(4 * units) + up256(2 * n * hq * hd) + 2 * up256(2 * hkv * n * hd)
        assert fa.prefill_workspace_bytes(n, hq, hkv, hd) == want, (n, hq, hkv, hd)
    pos0, n = 700, 1400
    units = -(-n // 128) * 32
    want = (256 + up256(4 * units) + up256(2 * n * 32 * 128)
            + 2 * up256(2 * 4 * (pos0 + n) * 128))
    assert fa.prefill_chunk_workspace_bytes(pos0, n, 32, 4, 128) == want
    d = fa.decode_workspace_bytes(32, 16, 256, 128)
    assert d >= 256 + 32 * 16 * 128 * (2 + 256) * 4
    assert fa.decode_workspace_bytes(0, 16, 256, 128) == 0
    assert fa.prefill_tile_shape(256) == (128, 128)
    with pytest.raises(fa.FAError):
        fa.prefill_tile_shape(96)


def _prefill_status(fa, **kw):
    args = dict(q=16, k=16, v=16, out=16, n=16, hq=8, hkv=2, hd=64, sink=0, win=0, fmt=0,
                max_seq=16, ss=0, sw=0, ws=16, wsb=1 << 30, tile_map=None)
    args.update(kw)
    L = fa.lib()
    return L.fa_prefill(args["q"], args["k"], args["v"], args["out"], args["n"], args["hq"],
                        args["hkv"], args["hd"], args["sink"], args["win"], args["fmt"],
                        args["max_seq"], args["ss"], args["sw"], args["ws"], args["wsb"],
                        args["tile_map"], None)


def test_prefill_validation(fa):
    assert _prefill_status(fa, hd=96) == fa.ERR_UNSUPPORTED
    assert _prefill_status(fa, hd=100) == fa.ERR_INVALID
    assert _prefill_status(fa, hq=6, hkv=4) == fa.ERR_INVALID
    assert _prefill_status(fa, hq=12, hkv=1) == fa.ERR_UNSUPPORTED   # group 12
    assert _prefill_status(fa, q=None) == fa.ERR_INVALID
    assert _prefill_status(fa, out=24) == fa.ERR_INVALID           # misaligned
    assert _prefill_status(fa, n=17, max_seq=16) == fa.ERR_INVALID
    assert _prefill_status(fa, sink=-1) == fa.ERR_INVALID
    assert _prefill_status(fa, fmt=7) == fa.ERR_INVALID            # no such format
    for fmt in (0, 2, 3):                                          # shadows only for Q4_0
        assert _prefill_status(fa, fmt=fmt, ss=4) == fa.ERR_INVALID
        assert _prefill_status(fa, fmt=fmt, sw=256) == fa.ERR_INVALID
    assert _prefill_status(fa, fmt=1, ss=9) == fa.ERR_INVALID
    assert _prefill_status(fa, fmt=1, sw=257) == fa.ERR_INVALID
    # a Q4_0 shadow window narrower than the ring runs the prefill in two parts
    # and needs the larger workspace
    plain = fa.prefill_workspace_bytes(16, 8, 2, 64)
    split = fa.prefill_workspace_bytes(16, 8, 2, 64, kv_fmt=1, shadow_win=100)
    assert split > plain
    assert _prefill_status(fa, fmt=1, sw=100, wsb=plain) == fa.ERR_WORKSPACE
    for fmt, sw in ((1, 0), (1, 256), (0, 0), (2, 0), (3, 0)):
        assert fa.prefill_workspace_bytes(16, 8, 2, 64, kv_fmt=fmt, shadow_win=sw) == plain
    assert _prefill_status(fa, wsb=10) == fa.ERR_WORKSPACE
    assert _prefill_status(fa, n=0) == fa.OK                       # empty input: nothing to do


def test_decode_and_append_validation(fa):
    L = fa.lib()
    # fa_decode(q, k, v, pos, nslots, hq, hkv, hd, max_seq, sink, win, fmt, ss, sw, kps, cap, ws, wsb, stream)
    base = [16, 16, 16, 16, 2, 16, 2, 256, 100, 0, 0, 1, 4, 0, 256, 4, 16, 1 << 30, None]

    def dec(**kw):
        a = list(base)
        for i, v in kw.items():
            a[int(i[1:])] = v
        return L.fa_decode(*a)
    assert dec(a14=0) == fa.ERR_INVALID        # split_keys
    assert dec(a15=0) == fa.ERR_INVALID        # max_splits
    assert dec(a3=None) == fa.ERR_INVALID      # pos
    assert dec(a3=18) == fa.ERR_INVALID        # pos misaligned
    assert dec(a17=100) == fa.ERR_WORKSPACE
    assert dec(a7=48) == fa.ERR_INVALID
    assert dec(a4=0) == fa.OK                  # no slots
    assert L.fa_decode_combine(16, 16, 2, 16, 256, 0, None) == fa.ERR_INVALID
    assert L.fa_decode_combine(16, 16, 2, 16, 96, 4, None) == fa.ERR_UNSUPPORTED
    # fa_kv_append(k, v, kp, vp, pos0, nslots, n, hkv, hd, max_seq, fmt, ss, sw, stream)
    assert L.fa_kv_append(16, 16, 16, 16, 16, 1, 8, 2, 64, 4, 1, 0, 0, None) == fa.ERR_INVALID
    assert L.fa_kv_append(16, 16, 16, 16, 16, 1, 8, 2, 64, 16, 0, 1, 0, None) == fa.ERR_INVALID
    assert L.fa_kv_append(16, 16, 16, 16, 16, 1, 8, 2, 96, 16, 1, 0, 0, None) == fa.ERR_UNSUPPORTED
    assert L.fa_kv_append(None, 16, 16, 16, 16, 1, 8, 2, 64, 16, 1, 0, 0, None) == fa.ERR_INVALID
    assert L.fa_kv_append(16, 16, 16, 16, 16, 0, 8, 2, 64, 16, 1, 0, 0, None) == fa.OK


def test_prefill_lse_and_merge_reject_bad_arguments(fa):
    L = fa.lib()
    # fa_prefill_lse: a misaligned lse pointer, and fa_prefill's own checks
    base = (16, 16, 16, 16)
    rest = (16, 8, 2, 64, 0, 0, 0, 16, 0, 0, 16, 1 << 30, None, None)
    assert L.fa_prefill_lse(*base, 18, *rest) == fa.ERR_INVALID
    bad_heads = (16, 8, 3, 64) + rest[4:]
    assert L.fa_prefill_lse(*base, None, *bad_heads) == fa.ERR_INVALID
    # n = 0 is a no-op
    assert L.fa_prefill_lse(*base, 16, 0, *rest[1:]) == fa.OK
    # fa_merge_attn_states: sizes, NULL inputs and alignment, before any launch
    def merge(out=16, out_lse=16, pre=16, pl=16, suf=16, sl=16, T=4, H=2, D=64, wc=-1):
        return L.fa_merge_attn_states(out, out_lse, pre, pl, suf, sl, T, H, D, wc, None)
    assert merge(D=6) == fa.ERR_INVALID
    assert merge(D=0) == fa.ERR_INVALID
    assert merge(H=0) == fa.ERR_INVALID
    assert merge(T=-1) == fa.ERR_INVALID
    assert merge(T=0) == fa.OK
    assert merge(pre=None) == fa.ERR_INVALID
    assert merge(sl=None) == fa.ERR_INVALID
    assert merge(out=8) == fa.ERR_INVALID
    assert merge(pl=18) == fa.ERR_INVALID
    assert merge(out_lse=2) == fa.ERR_INVALID


def test_f16_and_fp8_planes(fa):
    """fp16 rows of 2*hd bytes; fp8 rows of hd bytes plus a 256-byte block for
    the plane's fp32 scale right after the (256-rounded) body."""
    for hd in (64, 128, 256):
        row, body, sink, ring = fa.kv_plane_layout(fa.KV_F16, 2, 1000, hd)
        assert (row, body, sink, ring) == (2 * hd, 0, 0, 0)
        assert fa.kv_plane_bytes(fa.KV_F16, 2, 1000, hd) == ((2 * 1000 * 2 * hd + 255) // 256) * 256
        assert fa.kv_scale_offset(fa.KV_F16, 2, 1000, hd) == 0
        row, body, sink, ring = fa.kv_plane_layout(fa.KV_FP8_E4M3, 2, 1000, hd)
        assert (row, body, sink, ring) == (hd, 0, 0, 0)
        so = fa.kv_scale_offset(fa.KV_FP8_E4M3, 2, 1000, hd)
        assert so == ((2 * 1000 * hd + 255) // 256) * 256
        assert fa.kv_plane_bytes(fa.KV_FP8_E4M3, 2, 1000, hd) == so + 256
    assert fa.kv_scale_offset(fa.KV_Q4_0, 2, 1000, 64) == 0


def test_fp8_scale_and_narrow_format_validation(fa):
    L = fa.lib()
    # fa_kv_set_scale(planes, nslots, fmt, hkv, max_seq, hd, scale, stream)
    for bad in (0.0, -1.0, float("nan"), float("inf")):
        assert L.fa_kv_set_scale(16, 1, fa.KV_FP8_E4M3, 2, 64, 64, bad, None) == fa.ERR_INVALID
    assert L.fa_kv_set_scale(16, 1, fa.KV_F16, 2, 64, 64, 1.0, None) == fa.ERR_INVALID
    assert L.fa_kv_set_scale(None, 1, fa.KV_FP8_E4M3, 2, 64, 64, 1.0, None) == fa.ERR_INVALID
    assert L.fa_kv_set_scale(16, 0, fa.KV_FP8_E4M3, 2, 64, 64, 1.0, None) == fa.OK
    # the narrow formats have no fp16 shadows
    for fmt in (fa.KV_F16, fa.KV_FP8_E4M3):
        assert L.fa_kv_append(16, 16, 16, 16, 16, 1, 8, 2, 64, 16, fmt, 1, 0, None) == fa.ERR_INVALID
        assert L.fa_kv_append(16, 16, 16, 16, 16, 0, 8, 2, 64, 16, fmt, 0, 0, None) == fa.OK


def test_kv_init_validation(fa):
    L = fa.lib()
    # fa_kv_init(planes, nslots, fmt, hkv, max_seq, hd, shadow_sink, shadow_win, stream)
    assert L.fa_kv_init(16, 1, 7, 2, 64, 64, 0, 0, None) == fa.ERR_INVALID        # format
    assert L.fa_kv_init(16, 1, fa.KV_F32, 2, 64, 64, 4, 0, None) == fa.ERR_INVALID  # shadows
    assert L.fa_kv_init(16, 1, fa.KV_Q4_0, 2, 64, 64, 9, 0, None) == fa.ERR_INVALID
    assert L.fa_kv_init(16, 1, fa.KV_F16, 2, 64, 96, 0, 0, None) == fa.ERR_UNSUPPORTED
    assert L.fa_kv_init(None, 1, fa.KV_F16, 2, 64, 64, 0, 0, None) == fa.ERR_INVALID
    assert L.fa_kv_init(24, 1, fa.KV_F16, 2, 64, 64, 0, 0, None) == fa.ERR_INVALID   # misaligned
    assert L.fa_kv_init(16, 0, fa.KV_Q4_0, 2, 64, 64, 4, 256, None) == fa.OK         # no planes


def test_chunk_noalloc_layout_and_tile_shape_validation(fa):
    """Argument checks that return before any launch, and the plane layout and
    tile shape in closed form (include/fa.h)."""
    import ctypes
    L = fa.lib()

    def chunk(pos0=0, n=16, max_seq=32, wsb=1 << 30, q=16, lse=None):
        return L.fa_prefill_chunk(q, 16, 16, 16, lse, pos0, n, 8, 2, 64, 0, 0, 0, max_seq, 0, 0,
                                  16, wsb, None, None)
    assert chunk(pos0=-1) == fa.ERR_INVALID
    assert chunk(pos0=20, n=16) == fa.ERR_INVALID      # pos0 + n > max_seq
    assert chunk(wsb=10) == fa.ERR_WORKSPACE
    assert chunk(q=None) == fa.ERR_INVALID
    assert chunk(lse=18) == fa.ERR_INVALID             # misaligned lse
    assert chunk(n=0) == fa.OK                         # nothing to do

    def noalloc(nslots=2, hd=256, max_seq=100, kps=256, cap=4, pos=16):
        return L.fa_decode_noalloc(16, 16, 16, pos, nslots, 16, 2, hd, max_seq, 0, 0, 1, 4, 0,
                                   kps, cap, 16, None)
    assert noalloc(kps=0) == fa.ERR_INVALID
    assert noalloc(cap=0) == fa.ERR_INVALID
    assert noalloc(pos=None) == fa.ERR_INVALID
    assert noalloc(hd=96) == fa.ERR_UNSUPPORTED
    assert noalloc(nslots=0) == fa.OK
    # partials beyond the library's fixed 8 MiB array
    assert noalloc(nslots=4096, max_seq=1 << 20, cap=4096) == fa.ERR_WORKSPACE

    vals = [ctypes.c_size_t() for _ in range(4)]
    refs = [ctypes.byref(v) for v in vals]
    # Q4_0, 2 kv heads, 1024 rows, head_dim 256: 144-byte rows; the sink block
    # [2][8][256] fp16 after the body, the ring after the sinks (256-byte aligned)
    assert L.fa_kv_plane_layout(1, 2, 1024, 256, *refs) == fa.OK
    assert [v.value for v in vals] == [144, 0, 2 * 1024 * 144, 2 * 1024 * 144 + 2 * 8 * 256 * 2]
    assert L.fa_kv_plane_layout(2, 2, 1024, 128, *refs) == fa.OK  # fp16: rows only
    assert [v.value for v in vals[:2]] == [256, 0]
    assert L.fa_kv_plane_layout(1, 2, 1024, 100, *refs) == fa.ERR_INVALID
    bq, bk = ctypes.c_int(), ctypes.c_int()
    assert L.fa_prefill_tile_shape(256, ctypes.byref(bq), ctypes.byref(bk)) == fa.OK
    assert (bq.value, bk.value) == (128, 128)
    assert L.fa_prefill_tile_shape(96, ctypes.byref(bq), ctypes.byref(bk)) == fa.ERR_UNSUPPORTED
