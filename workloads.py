"""Seeded synthetic inputs and workload shapes for causal GQA flash attention.

This module is shared by the tests, the oracle checks and the benchmark. It
holds no attention arithmetic: it only draws random numbers and names shapes.

Recipe (the same everywhere):
  * seed = 20261202 + 1000 * workload_index (the index of the workload in
    WORKLOADS below); a numpy PCG64 stream;
  * draw order Q, then K, then V, each ``standard_normal`` in float64, cast
    to float32, in the logical order [n][heads][head_dim];
  * the multi-slot decode workload draws one slot at a time from the sub-seed
    seed + slot, in the order q[heads][head_dim], K[L][kv_heads][head_dim],
    V[L][kv_heads][head_dim].
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    index: int
    kind: str          # "prefill" or "decode"
    n: int             # prefill: tokens; decode: context length L per slot
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    sink: int          # attended set: sinks [0, sink)
    win: int           # attended set: recent window of win keys (<= 0: full causal)
    kv_fmt: str        # "f32", "q4_0", "f16" or "fp8_e4m3"
    shadow_sink: int = 0   # fp16 shadow geometry of a Q4_0 cache
    shadow_win: int = 0
    nslots: int = 1
    split_keys: int = 256
    k_scale: float = 1.0   # per-tensor scales of an fp8 cache (1.0: uncalibrated)
    v_scale: float = 1.0

    @property
    def seed(self) -> int:
        return SEED_BASE + 1000 * self.index


WORKLOADS = [
    Workload("prefill_f32_n128_h8x2_d64", 0, "prefill", 128, 8, 2, 64, 0, 0, "f32"),
    Workload("prefill_f32_n8192_h16x2_d256", 1, "prefill", 8192, 16, 2, 256, 0, 0, "f32"),
    Workload("prefill_f32_n8192_h16x2_d256_sink4_win1024", 2, "prefill", 8192, 16, 2, 256,
             4, 1024, "f32"),
    Workload("prefill_q4_n8192_h16x2_d256_shadow4_256", 3, "prefill", 8192, 16, 2, 256, 0, 0,
             "q4_0", shadow_sink=4, shadow_win=256),
    Workload("decode_q4_32slots_L32768_h16x2_d256_sink4", 4, "decode", 32768, 16, 2, 256, 4, 0,
             "q4_0", shadow_sink=4, shadow_win=0, nslots=32, split_keys=256),
    # the same shapes over the fp16 and fp8 e4m3fn cache formats
    Workload("prefill_f16_n8192_h16x2_d256", 5, "prefill", 8192, 16, 2, 256, 0, 0, "f16"),
    Workload("prefill_fp8_n8192_h16x2_d256", 6, "prefill", 8192, 16, 2, 256, 0, 0, "fp8_e4m3"),
    Workload("decode_f16_32slots_L32768_h16x2_d256_sink4", 7, "decode", 32768, 16, 2, 256, 4, 0,
             "f16", nslots=32, split_keys=256),
    Workload("decode_fp8_32slots_L32768_h16x2_d256_sink4", 8, "decode", 32768, 16, 2, 256, 4, 0,
             "fp8_e4m3", nslots=32, split_keys=256),
    # the windowed prefill over a Q4_0 cache with fp16 shadows (4 sinks, 256-row ring)
    Workload("prefill_q4_n8192_h16x2_d256_shadow4_256_sink4_win1024", 9, "prefill", 8192, 16, 2,
             256, 4, 1024, "q4_0", shadow_sink=4, shadow_win=256),
]

FMT_CODES = {"f32": 0, "q4_0": 1, "f16": 2, "fp8_e4m3": 3}  # include/fa.h FA_KV_*

BY_NAME = {w.name: w for w in WORKLOADS}


def _normal_f32(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(size=shape, dtype=np.float64).astype(np.float32)


def prefill_inputs(n: int, n_q_heads: int, n_kv_heads: int, head_dim: int, seed: int):
    """Q [n][Hq][hd], K [n][Hkv][hd], V [n][Hkv][hd], float32, drawn Q, K, V."""
    rng = np.random.Generator(np.random.PCG64(seed))
    q = _normal_f32(rng, (n, n_q_heads, head_dim))
    k = _normal_f32(rng, (n, n_kv_heads, head_dim))
    v = _normal_f32(rng, (n, n_kv_heads, head_dim))
    return q, k, v


def decode_slot_inputs(L: int, n_q_heads: int, n_kv_heads: int, head_dim: int, seed: int,
                       slot: int):
    """One decode slot: q [Hq][hd], K [L][Hkv][hd], V [L][Hkv][hd] from seed + slot."""
    rng = np.random.Generator(np.random.PCG64(seed + slot))
    q = _normal_f32(rng, (n_q_heads, head_dim))
    k = _normal_f32(rng, (L, n_kv_heads, head_dim))
    v = _normal_f32(rng, (L, n_kv_heads, head_dim))
    return q, k, v


def workload_inputs(w: Workload):
    if w.kind == "prefill":
        return prefill_inputs(w.n, w.n_q_heads, w.n_kv_heads, w.head_dim, w.seed)
    raise ValueError("decode workloads are drawn per slot with decode_slot_inputs")
