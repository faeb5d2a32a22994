"""numpy front end of the C oracle (oracle.c).

Test infrastructure: only the tests, the smoke check and the benchmark's CPU
baseline use it. Every function follows a definition on the pages:

* ``f16_rne`` / ``f16_to_f64``: binary16 round-to-nearest-even and its exact
  value ("attention.cu", fc_attn_kv_append_q4: rows mirrored with __float2half).
* ``q4_encode`` / ``q4_decode``: the Q4_0 block format ("attention.cu",
  "4-bit KV cache (Q4_0 blocks)", fc_kvq4_quant_block, fc_kvq4_dequant_elem).
* ``visible`` / ``tile_map``: the attended key set with sinks and a recent
  window ("attention.cu" file header, fc_attn_tile_in_window), and the
  brute-force map of key tiles a query tile must visit.
* ``reads_fp16``: which copy of a key a Q4_0 reader sees ("attention.cu",
  fc_kvq4_is_fp16 and the ring liveness floor in fc_attn_flash_prefill_q4).
* ``attention``: softmax(scale q k^T) v over the attended set, fp64, two-pass
  global max ("vt/ops.h" vt::Attention; "qwen38_batched.rs" bq_attn).
* ``dec_plan`` / ``partial`` / ``combine``: split-KV decode partials and their
  log-sum-exp merge ("attention.cu", "Decode-mode flash attention").
"""
from __future__ import annotations

import ctypes
import math
import os

import numpy as np

from . import build as _build

RING_ROWS = 256
SINK_MAX = 8
Q4_BLOCK = 32
Q4_BLOCK_BYTES = 18

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        L.oracle_f16_rne.restype = ctypes.c_uint16
        L.oracle_f16_rne.argtypes = [ctypes.c_float]
        L.oracle_f16_to_f64.restype = f64
        L.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        L.oracle_f16_rne_array.argtypes = [P, i64, P]
        L.oracle_f16_to_f64_array.argtypes = [P, i64, P]
        L.oracle_e4m3_rne_sat.restype = ctypes.c_uint8
        L.oracle_e4m3_rne_sat.argtypes = [ctypes.c_float]
        L.oracle_e4m3_to_f64.restype = f64
        L.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        L.oracle_e4m3_store_array.argtypes = [P, i64, ctypes.c_float, P]
        L.oracle_e4m3_load_array.argtypes = [P, i64, ctypes.c_float, P]
        L.oracle_q4_encode_block.argtypes = [P, P]
        L.oracle_q4_decode_block.argtypes = [P, P]
        L.oracle_q4_encode_rows.argtypes = [P, i64, i32, P]
        L.oracle_q4_decode_rows.argtypes = [P, i64, i32, P]
        L.oracle_visible.restype = i32
        L.oracle_visible.argtypes = [i32, i32, i32, i32]
        L.oracle_tile_map.argtypes = [i32, i32, i32, i32, i32, i32, P]
        L.oracle_reads_fp16.restype = i32
        L.oracle_reads_fp16.argtypes = [i32, i32, i32, i32, i32]
        L.oracle_attention.restype = i32
        L.oracle_attention.argtypes = [P, P, i32, i32, i32, i32, i32, P, P, P, P,
                                       i32, i32, i32, i32, f64, P, P]
        L.oracle_merge_attn_states.restype = None
        L.oracle_merge_attn_states.argtypes = [P, P, P, P, i32, i32, i32, i32, P, P]
        L.oracle_dec_plan.restype = i32
        L.oracle_dec_plan.argtypes = [i32, i32, i32, ctypes.POINTER(i32)]
        L.oracle_partial.argtypes = [P, i32, i32, i32, i32, i32, i32, i32, P, P, P, P,
                                     i32, i32, i32, i32, f64, P, P, P]
        L.oracle_combine.restype = i32
        L.oracle_combine.argtypes = [P, P, P, i32, i32, P]
        L.oracle_num_threads.restype = i32
        _lib = L
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def num_threads() -> int:
    return int(lib().oracle_num_threads())


# ---------------------------------------------------------------- fp16

def f16_rne(x) -> np.ndarray:
    """float32 array -> uint16 binary16 bits, round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint16)
    lib().oracle_f16_rne_array(_ptr(x), x.size, _ptr(out))
    return out


def f16_to_f64(h) -> np.ndarray:
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, np.float64)
    lib().oracle_f16_to_f64_array(_ptr(h), h.size, _ptr(out))
    return out


# ---------------------------------------------------------- fp8 e4m3fn

def e4m3(x: float) -> int:
    """One float -> e4m3fn byte, round to nearest even, saturating at +-448."""
    return int(lib().oracle_e4m3_rne_sat(float(np.float32(x))))


def e4m3_value(code: int) -> float:
    return float(lib().oracle_e4m3_to_f64(int(code) & 0xff))


def e4m3_store(x, scale: float) -> np.ndarray:
    """The fp8 KV store: bytes of Quantize(x / scale), elementwise."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, np.uint8)
    lib().oracle_e4m3_store_array(_ptr(x), x.size, float(np.float32(scale)), _ptr(out))
    return out


def e4m3_load(q, scale: float) -> np.ndarray:
    """The fp8 KV read: Dequant(byte) * scale in float, as float64."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    out = np.empty(q.shape, np.float64)
    lib().oracle_e4m3_load_array(_ptr(q), q.size, float(np.float32(scale)), _ptr(out))
    return out


# ---------------------------------------------------------------- Q4_0

def q4_encode(x) -> np.ndarray:
    """[..., hd] float32 rows -> [..., hd/32*18] uint8 Q4_0 rows."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    hd = x.shape[-1]
    if hd % Q4_BLOCK:
        raise ValueError("head_dim must be a multiple of 32")
    rows = x.size // hd
    out = np.empty(x.shape[:-1] + (hd // Q4_BLOCK * Q4_BLOCK_BYTES,), np.uint8)
    lib().oracle_q4_encode_rows(_ptr(x), rows, hd, _ptr(out))
    return out


def q4_decode(b, head_dim: int) -> np.ndarray:
    """[..., hd/32*18] uint8 rows -> [..., hd] float64 exact values."""
    b = np.ascontiguousarray(b, dtype=np.uint8)
    rb = head_dim // Q4_BLOCK * Q4_BLOCK_BYTES
    if b.shape[-1] != rb:
        raise ValueError("row bytes do not match head_dim")
    rows = b.size // rb
    out = np.empty(b.shape[:-1] + (head_dim,), np.float64)
    lib().oracle_q4_decode_rows(_ptr(b), rows, head_dim, _ptr(out))
    return out


# ----------------------------------------------------------- visibility

def visible(p: int, j: int, sink: int, win: int) -> bool:
    return bool(lib().oracle_visible(p, j, sink, win))


def tile_map(n: int, bq: int, bk: int, sink: int, win: int, pos0: int = 0) -> np.ndarray:
    """[ceil(n/bq)][ceil((pos0+n)/bk)] visited (query tile, key tile) pairs of n
    queries at positions pos0.. over keys 0..pos0+n-1."""
    nqt, nkt = -(-n // bq), -(-(pos0 + n) // bk)
    out = np.zeros((nqt, nkt), np.uint8)
    lib().oracle_tile_map(pos0, n, bq, bk, sink, win, _ptr(out))
    return out


def reads_fp16(p: int, s: int, L: int, shadow_sink: int, shadow_win: int) -> bool:
    return bool(lib().oracle_reads_fp16(p, s, L, shadow_sink, shadow_win))


# ------------------------------------------------------------ KV values

class KVValues:
    """The values a reader of one KV cache sees, [L][Hkv][hd] float64.

    ``body`` is the main store: fp32 widened, the fp16 rounding ("f16"), the
    fp8 e4m3fn store and read with the tensor's scale ("fp8_e4m3"), or Q4_0
    decoded. ``f16`` is the fp16 shadow copy of every row of a Q4_0 cache (None
    otherwise); ``q4`` / ``fp8`` the bytes the oracle stored."""

    def __init__(self, x_f32: np.ndarray, kv_fmt: str, scale: float = 1.0):
        x_f32 = np.ascontiguousarray(x_f32, dtype=np.float32)
        self.kv_fmt = kv_fmt
        self.f16 = None
        self.q4 = None
        self.fp8 = None
        if kv_fmt == "f32":
            self.body = x_f32.astype(np.float64)
        elif kv_fmt == "f16":
            self.body = f16_to_f64(f16_rne(x_f32))
        elif kv_fmt == "fp8_e4m3":
            self.fp8 = e4m3_store(x_f32, scale)
            self.body = e4m3_load(self.fp8, scale)
        elif kv_fmt == "q4_0":
            self.q4 = q4_encode(x_f32)
            self.body = q4_decode(self.q4, x_f32.shape[-1])
            self.f16 = f16_to_f64(f16_rne(x_f32))
        else:
            raise ValueError(kv_fmt)


def attention(q, qpos, kv_k: KVValues, kv_v: KVValues, *, sink: int, win: int,
              shadow_sink: int = 0, shadow_win: int = 0, scale: float | None = None,
              L: int | None = None, with_lse: bool = False):
    """out [nq][Hq][hd] float64 for query rows q [nq][Hq][hd] at positions qpos;
    with with_lse, also lse [nq][Hq] = log sum_j exp(s_j) of each row's scores.

    L is the number of rows in the cache (last appended row L-1), which decides
    the fp16 ring liveness of a Q4_0 cache; it defaults to the cache size."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    qpos = np.ascontiguousarray(qpos, dtype=np.int32)
    nq, Hq, hd = q.shape
    Lc, Hkv, hd2 = kv_k.body.shape
    assert hd2 == hd and qpos.shape == (nq,)
    if L is None:
        L = Lc
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    out = np.empty((nq, Hq, hd), np.float64)
    lse = np.empty((nq, Hq), np.float64) if with_lse else None
    kf = kv_k.f16 if kv_k.f16 is not None else None
    vf = kv_v.f16 if kv_v.f16 is not None else None
    st = lib().oracle_attention(
        _ptr(q), _ptr(qpos), nq, Hq, Hkv, hd, L, _ptr(kv_k.body), _ptr(kv_v.body),
        _ptr(kf) if kf is not None else None, _ptr(vf) if vf is not None else None,
        shadow_sink, shadow_win, sink, win, float(scale), _ptr(out),
        _ptr(lse) if lse is not None else None)
    if st != 0:
        raise ValueError(f"oracle_attention failed with status {st}")
    return (out, lse) if with_lse else out


def prefill(q, k, v, *, kv_fmt: str, sink: int, win: int, shadow_sink: int = 0,
            shadow_win: int = 0, rows=None, with_lse: bool = False, pos0: int = 0,
            k_scale: float = 1.0, v_scale: float = 1.0):
    """Prefill of n queries at positions pos0 .. pos0+n-1 (query t at pos0 + t)
    over the cache rows 0 .. pos0+n-1: q [n][Hq][hd], k, v [pos0+n][Hkv][hd].

    rows selects query rows t (default all); returns [len(rows)][Hq][hd], and
    with with_lse also the rows' lse [len(rows)][Hq]."""
    n = q.shape[0]
    L = pos0 + n
    assert k.shape[0] >= L and v.shape[0] >= L
    if rows is None:
        rows = np.arange(n, dtype=np.int32)
    rows = np.asarray(rows, dtype=np.int32)
    kk, vv = KVValues(k[:L], kv_fmt, k_scale), KVValues(v[:L], kv_fmt, v_scale)
    return attention(q[rows], rows + pos0, kk, vv, sink=sink, win=win, shadow_sink=shadow_sink,
                     shadow_win=shadow_win, L=L, with_lse=with_lse)


def merge_attn_states(prefix, prefix_lse, suffix, suffix_lse, with_context: int = -1):
    """[B] MergeAttnStates on float32 inputs: outputs [T][H][D], lses [H][T].

    Returns (out [T][H][D], out_lse [H][T]) in float64; tokens t >=
    with_context (when >= 0) take the suffix unchanged."""
    prefix = np.ascontiguousarray(prefix, dtype=np.float32)
    suffix = np.ascontiguousarray(suffix, dtype=np.float32)
    prefix_lse = np.ascontiguousarray(prefix_lse, dtype=np.float32)
    suffix_lse = np.ascontiguousarray(suffix_lse, dtype=np.float32)
    T, H, D = prefix.shape
    assert suffix.shape == (T, H, D) and prefix_lse.shape == (H, T) == suffix_lse.shape
    out = np.empty((T, H, D), np.float64)
    out_lse = np.empty((H, T), np.float64)
    lib().oracle_merge_attn_states(_ptr(prefix), _ptr(prefix_lse), _ptr(suffix),
                                   _ptr(suffix_lse), T, H, D, int(with_context), _ptr(out),
                                   _ptr(out_lse))
    return out, out_lse


# ------------------------------------------------- split-KV decode + merge

def dec_plan(seq_len: int, kps: int, cap: int):
    """(live splits, split_len) of the decode split plan."""
    sl = ctypes.c_int(0)
    ns = lib().oracle_dec_plan(seq_len, kps, cap, ctypes.byref(sl))
    return int(ns), int(sl.value)


def partial(q, p: int, k_lo: int, k_hi: int, kv_k: KVValues, kv_v: KVValues, *, sink: int,
            win: int, shadow_sink: int = 0, shadow_win: int = 0, L: int | None = None,
            scale: float | None = None):
    """Unnormalised (m [Hq], l [Hq], acc [Hq][hd]) over keys [k_lo, k_hi) for q [Hq][hd]."""
    q = np.ascontiguousarray(q, dtype=np.float32)
    Hq, hd = q.shape
    Lc, Hkv, _ = kv_k.body.shape
    if L is None:
        L = Lc
    if scale is None:
        scale = 1.0 / math.sqrt(hd)
    m = np.empty(Hq, np.float64)
    l = np.empty(Hq, np.float64)
    acc = np.empty((Hq, hd), np.float64)
    kf = kv_k.f16 if kv_k.f16 is not None else None
    vf = kv_v.f16 if kv_v.f16 is not None else None
    lib().oracle_partial(_ptr(q), p, k_lo, k_hi, Hq, Hkv, hd, L, _ptr(kv_k.body),
                         _ptr(kv_v.body), _ptr(kf) if kf is not None else None,
                         _ptr(vf) if vf is not None else None, shadow_sink, shadow_win, sink,
                         win, float(scale), _ptr(m), _ptr(l), _ptr(acc))
    return m, l, acc


def combine(m, l, acc) -> np.ndarray:
    """Merge ns partials of one head: m [ns], l [ns], acc [ns][hd] -> out [hd]."""
    m = np.ascontiguousarray(m, dtype=np.float64)
    l = np.ascontiguousarray(l, dtype=np.float64)
    acc = np.ascontiguousarray(acc, dtype=np.float64)
    ns, hd = acc.shape
    out = np.empty(hd, np.float64)
    if lib().oracle_combine(_ptr(m), _ptr(l), _ptr(acc), ns, hd, _ptr(out)) != 0:
        raise ValueError("every split is empty")
    return out


def decode(q, pos: int, k, v, *, kv_fmt: str, sink: int, win: int, shadow_sink: int = 0,
           shadow_win: int = 0, k_scale: float = 1.0, v_scale: float = 1.0) -> np.ndarray:
    """One decode query q [Hq][hd] at position pos over rows 0..pos of K, V [L][Hkv][hd]."""
    kk = KVValues(np.ascontiguousarray(k[: pos + 1]), kv_fmt, k_scale)
    vv = KVValues(np.ascontiguousarray(v[: pos + 1]), kv_fmt, v_scale)
    out = attention(q[None], np.array([pos], np.int32), kk, vv, sink=sink, win=win,
                    shadow_sink=shadow_sink, shadow_win=shadow_win, L=pos + 1)
    return out[0]
