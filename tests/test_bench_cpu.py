"""The work counts behind the benchmark's throughput figures, on the CPU.

A TFLOP/s or GB/s number is only as good as the work it divides: the attended
(query, key) pairs of a prefill (4 * head_dim * n_q_heads flop each) and the KV
bytes a decode step must read."""
import importlib.util
import os

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


@pytest.mark.parametrize("sink,win", [(0, 0), (0, 1), (4, 0), (4, 1), (4, 16), (9, 3), (0, 40),
                                      (2, 100)])
def test_visible_pairs_is_the_brute_force_count(bench, oracle_mod, sink, win):
    for n in (1, 2, 17, 64):
        brute = sum(oracle_mod.visible(p, j, sink, win) for p in range(n) for j in range(p + 1))
        assert bench.visible_pairs(n, sink, win) == brute, (n, sink, win)


def test_full_causal_and_chunk_counts(bench):
    n = 8192
    assert bench.visible_pairs(n, 0, 0) == n * (n + 1) // 2
    # the chunk of queries 4096..8191 attends exactly the pairs the whole
    # prefill adds after its first 4096 queries
    chunk = sum(p + 1 for p in range(4096, 8192))
    assert bench.visible_pairs(8192, 0, 0) - bench.visible_pairs(4096, 0, 0) == chunk
    # a window of win keys and no sinks: min(p + 1, win) keys per query
    assert bench.visible_pairs(100, 0, 10) == sum(min(p + 1, 10) for p in range(100))


def test_decode_kv_bytes(bench):
    from workloads import BY_NAME
    w = BY_NAME["decode_q4_32slots_L32768_h16x2_d256_sink4"]
    # per (slot, kv head): 4 fp16 sink rows of K and V (512 bytes each) and the
    # other 32764 rows as Q4_0 K and V (144 bytes each)
    per = 4 * 2 * 512 + (32768 - 4) * 2 * 144
    assert bench.decode_kv_bytes(w) == 32 * 2 * per
    w16 = BY_NAME["decode_f16_32slots_L32768_h16x2_d256_sink4"]
    assert bench.decode_kv_bytes(w16) == 32 * 2 * 32768 * 2 * 512
    w8 = BY_NAME["decode_fp8_32slots_L32768_h16x2_d256_sink4"]
    assert bench.decode_kv_bytes(w8) == 32 * 2 * 32768 * 2 * 256


def test_append_q4_bytes(bench, oracle_mod):
    import numpy as np
    from workloads import BY_NAME
    w = BY_NAME["prefill_q4_n8192_h16x2_d256_shadow4_256"]
    rows = np.zeros((w.n, w.n_kv_heads, w.head_dim), np.float32)
    read = 2 * rows.nbytes                                  # K and V fp32 rows
    body = 2 * oracle_mod.q4_encode(rows).nbytes            # their Q4_0 blocks
    shadows = 2 * (4 + 256) * w.n_kv_heads * w.head_dim * 2  # fp16 sinks and ring
    assert bench.append_q4_bytes(w) == read + body + shadows == 38805504


def test_job_throughput_counts_every_rank(bench):
    # two replicas each doing 1e12 flop in 1 ms: 2e15 flop/s for the job
    assert bench.job_throughput(1e12, 1.0, 2) == pytest.approx(2e15)
