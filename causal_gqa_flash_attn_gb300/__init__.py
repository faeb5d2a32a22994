"""Causal grouped-query flash attention for GB300 (sm_103a).

A thin ctypes binding of libfa.so (C ABI in include/fa.h). Every function
takes torch tensors that already live on the GPU, checks dtype/contiguity,
passes raw pointers and the current CUDA stream, and raises FAError on a
non-OK status. All arithmetic runs in the library's CUDA kernels; there is no
CPU fallback, and importing this package fails if the library was not built
(run ``python -m causal_gqa_flash_attn_gb300.build`` or
``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libfa.so")

KV_F32 = 0
KV_Q4_0 = 1
KV_F16 = 2
KV_FP8_E4M3 = 3
Q4_SINK_MAX = 8
Q4_RING_ROWS = 256

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE, ERR_TIMEOUT, ERR_WORKSPACE = range(7)

# Public entry points of include/fa.h with their ctypes signatures.
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "fa_kv_plane_bytes": (_SZ, [_I, _I, _I, _I]),
    "fa_kv_plane_layout": (_I, [_I, _I, _I, _I, _P, _P, _P, _P]),
    "fa_kv_init": (_I, [_P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "fa_kv_scale_offset": (_SZ, [_I, _I, _I, _I]),
    "fa_kv_set_scale": (_I, [_P, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "fa_kv_append": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "fa_prefill_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "fa_prefill_tile_shape": (_I, [_I, _P, _P]),
    "fa_prefill": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _SZ, _P,
                        _P]),
    "fa_prefill_lse": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _SZ,
                            _P, _P]),
    "fa_merge_attn_states": (_I, [_P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _P]),
    "fa_prefill_chunk_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "fa_prefill_chunk_workspace_bytes_for": (_SZ, [_I, _I, _I, _I, _I, _I, _I]),
    "fa_prefill_chunk": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P,
                              _SZ, _P, _P]),
    "fa_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "fa_decode": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P, _SZ,
                       _P]),
    "fa_decode_combine": (_I, [_P, _P, _I, _I, _I, _I, _P]),
    "fa_decode_noalloc": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I, _I,
                               _P, _P]),
    "fa_set_kernel_events": (_I, [_P, _P]),
    "fa_get_device_error": (_I, [_P]),
    "fa_status_string": (ctypes.c_char_p, [_I]),
    "fa_version": (_I, []),
}


class FAError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libfa.so; raises ImportError if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libfa.so not built ({LIB_PATH}); run "
                              "python -m causal_gqa_flash_attn_gb300.build")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().fa_status_string(status).decode()


def _check(status: int, what: str):
    if status != OK:
        raise FAError(status, what)


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dev(t: torch.Tensor | None, dtype, name: str):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


# ------------------------------------------------------------------ planes

def kv_plane_bytes(kv_fmt: int, n_kv_heads: int, max_seq: int, head_dim: int) -> int:
    return int(lib().fa_kv_plane_bytes(kv_fmt, n_kv_heads, max_seq, head_dim))


def kv_plane_layout(kv_fmt: int, n_kv_heads: int, max_seq: int, head_dim: int):
    """(row_bytes, body_offset, sink_offset, ring_offset) of one plane."""
    vals = [ctypes.c_size_t(0) for _ in range(4)]
    _check(lib().fa_kv_plane_layout(kv_fmt, n_kv_heads, max_seq, head_dim,
                                    *[ctypes.byref(v) for v in vals]), "fa_kv_plane_layout")
    return tuple(int(v.value) for v in vals)


def kv_scale_offset(kv_fmt: int, n_kv_heads: int, max_seq: int, head_dim: int) -> int:
    """Byte offset of an fp8 plane's fp32 scale (0 for the other formats)."""
    return int(lib().fa_kv_scale_offset(kv_fmt, n_kv_heads, max_seq, head_dim))


def kv_set_scale(planes, kv_fmt: int, n_kv_heads: int, max_seq: int, head_dim: int,
                 scale: float, stream=None):
    """Set the scale of every fp8 plane in ``planes`` (consecutive planes)."""
    pb = kv_plane_bytes(kv_fmt, n_kv_heads, max_seq, head_dim)
    if pb == 0 or planes.numel() % pb:
        raise ValueError("planes is not a whole number of planes of this geometry")
    _check(lib().fa_kv_set_scale(_dev(planes, torch.uint8, "planes"), planes.numel() // pb,
                                 kv_fmt, n_kv_heads, max_seq, head_dim, float(scale),
                                 _stream(stream)), "fa_kv_set_scale")


def kv_init(planes, kv_fmt: int, n_kv_heads: int, max_seq: int, head_dim: int,
            shadow_sink: int = 0, shadow_win: int = 0, stream=None):
    """fa_kv_init over every plane in ``planes`` (consecutive planes)."""
    pb = kv_plane_bytes(kv_fmt, n_kv_heads, max_seq, head_dim)
    if pb == 0 or planes.numel() % pb:
        raise ValueError("planes is not a whole number of planes of this geometry")
    _check(lib().fa_kv_init(_dev(planes, torch.uint8, "planes"), planes.numel() // pb, kv_fmt,
                            n_kv_heads, max_seq, head_dim, shadow_sink, shadow_win,
                            _stream(stream)), "fa_kv_init")


def alloc_planes(nslots: int, kv_fmt: int, n_kv_heads: int, max_seq: int, head_dim: int,
                 device="cuda", scale: float = 1.0) -> torch.Tensor:
    """nslots consecutive planes as one uint8 tensor, prepared by fa_kv_init;
    fp8 planes get ``scale`` (the per-tensor k_scale or v_scale, 1.0
    uncalibrated)."""
    pb = kv_plane_bytes(kv_fmt, n_kv_heads, max_seq, head_dim)
    if pb == 0:
        raise ValueError("invalid plane geometry")
    planes = torch.empty(nslots * pb, dtype=torch.uint8, device=device)
    kv_init(planes, kv_fmt, n_kv_heads, max_seq, head_dim)
    if kv_fmt == KV_FP8_E4M3 and scale != 1.0:
        kv_set_scale(planes, kv_fmt, n_kv_heads, max_seq, head_dim, scale)
    return planes


def kv_append(k_new, v_new, k_planes, v_planes, pos0, *, n_kv_heads: int, head_dim: int,
              max_seq: int, kv_fmt: int, shadow_sink: int = 0, shadow_win: int = 0,
              stream=None):
    """Append k_new/v_new [nslots][n][n_kv_heads][head_dim] fp32 at pos0[slot] (int32)."""
    nslots, n = k_new.shape[0], k_new.shape[1]
    _check(lib().fa_kv_append(
        _dev(k_new, torch.float32, "k_new"), _dev(v_new, torch.float32, "v_new"),
        _dev(k_planes, torch.uint8, "k_planes"), _dev(v_planes, torch.uint8, "v_planes"),
        _dev(pos0, torch.int32, "pos0"), nslots, n, n_kv_heads, head_dim, max_seq, kv_fmt,
        shadow_sink, shadow_win, _stream(stream)), "fa_kv_append")


# ----------------------------------------------------------------- prefill

def prefill_workspace_bytes(n: int, n_q_heads: int, n_kv_heads: int, head_dim: int,
                            kv_fmt: int | None = None, shadow_win: int = 0) -> int:
    """Workspace of fa_prefill; pass kv_fmt and shadow_win to size a Q4_0 cache
    whose shadow window is neither 0 nor the whole ring."""
    if kv_fmt is not None:
        return prefill_chunk_workspace_bytes(0, n, n_q_heads, n_kv_heads, head_dim, kv_fmt,
                                             shadow_win)
    return int(lib().fa_prefill_workspace_bytes(n, n_q_heads, n_kv_heads, head_dim))


def prefill_tile_shape(head_dim: int):
    bq, bk = ctypes.c_int(0), ctypes.c_int(0)
    _check(lib().fa_prefill_tile_shape(head_dim, ctypes.byref(bq), ctypes.byref(bk)),
           "fa_prefill_tile_shape")
    return bq.value, bk.value


def prefill(q, k, v, out, n: int, n_q_heads: int, n_kv_heads: int, head_dim: int, sink: int,
            win: int, kv_fmt: int, *, max_seq: int, shadow_sink: int = 0, shadow_win: int = 0,
            workspace: torch.Tensor, tile_map: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, stream=None):
    """fa_prefill (fa_prefill_lse when lse [Hq][n] fp32 is given): q/out
    [n][Hq][hd] fp32, k/v one plane each (uint8 tensors)."""
    args = (_dev(q, torch.float32, "q"), _dev(k, torch.uint8, "k"), _dev(v, torch.uint8, "v"),
            _dev(out, torch.float32, "out"))
    rest = (n, n_q_heads, n_kv_heads, head_dim, sink, win, kv_fmt, max_seq, shadow_sink,
            shadow_win, _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
            _dev(tile_map, torch.uint8, "tile_map"), _stream(stream))
    if lse is None:
        _check(lib().fa_prefill(*args, *rest), "fa_prefill")
    else:
        _check(lib().fa_prefill_lse(*args, _dev(lse, torch.float32, "lse"), *rest),
               "fa_prefill_lse")


def prefill_chunk_workspace_bytes(pos0: int, n: int, n_q_heads: int, n_kv_heads: int,
                                  head_dim: int, kv_fmt: int | None = None,
                                  shadow_win: int = 0) -> int:
    if kv_fmt is not None:
        return int(lib().fa_prefill_chunk_workspace_bytes_for(pos0, n, n_q_heads, n_kv_heads,
                                                              head_dim, kv_fmt, shadow_win))
    return int(lib().fa_prefill_chunk_workspace_bytes(pos0, n, n_q_heads, n_kv_heads, head_dim))


def prefill_chunk(q, k, v, out, pos0: int, n: int, n_q_heads: int, n_kv_heads: int,
                  head_dim: int, sink: int, win: int, kv_fmt: int, *, max_seq: int,
                  shadow_sink: int = 0, shadow_win: int = 0, workspace: torch.Tensor,
                  tile_map: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                  stream=None):
    """fa_prefill_chunk: n queries at positions pos0.. over cache rows 0..pos0+n-1."""
    _check(lib().fa_prefill_chunk(
        _dev(q, torch.float32, "q"), _dev(k, torch.uint8, "k"), _dev(v, torch.uint8, "v"),
        _dev(out, torch.float32, "out"), _dev(lse, torch.float32, "lse"), pos0, n, n_q_heads,
        n_kv_heads, head_dim, sink, win, kv_fmt, max_seq, shadow_sink, shadow_win,
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _dev(tile_map, torch.uint8, "tile_map"), _stream(stream)), "fa_prefill_chunk")


def merge_attn_states(out, out_lse, prefix, prefix_lse, suffix, suffix_lse, *,
                      prefill_tokens_with_context: int = -1, stream=None):
    """fa_merge_attn_states: outputs [T][H][D] fp32, lses [H][T] fp32 (out_lse may be None)."""
    T, H, D = prefix.shape
    _check(lib().fa_merge_attn_states(
        _dev(out, torch.float32, "out"), _dev(out_lse, torch.float32, "out_lse"),
        _dev(prefix, torch.float32, "prefix"), _dev(prefix_lse, torch.float32, "prefix_lse"),
        _dev(suffix, torch.float32, "suffix"), _dev(suffix_lse, torch.float32, "suffix_lse"),
        T, H, D, prefill_tokens_with_context, _stream(stream)), "fa_merge_attn_states")


# ------------------------------------------------------------------ decode

def decode_workspace_bytes(nslots: int, n_q_heads: int, head_dim: int, max_splits: int) -> int:
    return int(lib().fa_decode_workspace_bytes(nslots, n_q_heads, head_dim, max_splits))


def decode(q, k_planes, v_planes, pos, *, n_q_heads: int, n_kv_heads: int, head_dim: int,
           max_seq: int, sink: int, win: int, kv_fmt: int, shadow_sink: int = 0,
           shadow_win: int = 0, split_keys: int = 256, max_splits: int, workspace: torch.Tensor,
           stream=None):
    """fa_decode: q [nslots][Hq][hd] fp32, pos [nslots] int32 (device)."""
    nslots = q.shape[0]
    _check(lib().fa_decode(
        _dev(q, torch.float32, "q"), _dev(k_planes, torch.uint8, "k_planes"),
        _dev(v_planes, torch.uint8, "v_planes"), _dev(pos, torch.int32, "pos"), nslots,
        n_q_heads, n_kv_heads, head_dim, max_seq, sink, win, kv_fmt, shadow_sink, shadow_win,
        split_keys, max_splits, _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)), "fa_decode")


def decode_combine(workspace, out, *, nslots: int, n_q_heads: int, head_dim: int,
                   max_splits: int, stream=None):
    _check(lib().fa_decode_combine(
        _dev(workspace, torch.uint8, "workspace"), _dev(out, torch.float32, "out"), nslots,
        n_q_heads, head_dim, max_splits, _stream(stream)), "fa_decode_combine")


def decode_noalloc(q, k_planes, v_planes, pos, out, *, n_q_heads: int, n_kv_heads: int,
                   head_dim: int, max_seq: int, sink: int, win: int, kv_fmt: int,
                   shadow_sink: int = 0, shadow_win: int = 0, split_keys: int = 256,
                   max_splits: int, stream=None):
    """fa_decode_noalloc: decode + combine into out [nslots][Hq][hd] with the
    partials in the library's fixed device array; for callers that cannot
    allocate device memory. Calls that overlap on the GPU race on that array."""
    nslots = q.shape[0]
    _check(lib().fa_decode_noalloc(
        _dev(q, torch.float32, "q"), _dev(k_planes, torch.uint8, "k_planes"),
        _dev(v_planes, torch.uint8, "v_planes"), _dev(pos, torch.int32, "pos"), nslots,
        n_q_heads, n_kv_heads, head_dim, max_seq, sink, win, kv_fmt, shadow_sink, shadow_win,
        split_keys, max_splits, _dev(out, torch.float32, "out"), _stream(stream)),
        "fa_decode_noalloc")


def set_kernel_events(start, stop):
    """Record torch.cuda.Event pair around the next tensor-core prefill /
    split-decode kernels (None, None to stop). Events must have been recorded
    once so that they exist."""
    h = lambda e: None if e is None else int(e.cuda_event)
    _check(lib().fa_set_kernel_events(h(start), h(stop)), "fa_set_kernel_events")


def get_device_error(stream=None) -> int:
    """Synchronise the stream; return (and clear) the device status."""
    return int(lib().fa_get_device_error(_stream(stream)))


def version() -> int:
    return int(lib().fa_version())
