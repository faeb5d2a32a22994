"""The operand precision of the tensor-core MMAs, decided on the CPU.

The attention kernels run QK^T and PV as MMAs whose inputs are 16-bit floats
with fp32 accumulation, fp32 softmax state and an fp32 output. Two 16-bit
formats feed the same MMA instruction at the same rate: bf16 (8 significant
bits) and binary16 (11). This test runs a rounding model of the kernels'
arithmetic on the CPU - fp64 attention in which q, k, v and the softmax
weights p are first rounded to the format - on heads shaped like the
8192-token workloads (16 q heads, 2 kv heads, head_dim 256, N(0,1) inputs,
full causal) at n = 512, and compares it with the oracle under the
tolerance every parity test uses (max-abs 5e-3, relative L2 2e-3).

bf16 fails that tolerance: the first query attends to key 0 alone, so its
output is v_0 rounded, and for |v| in [2, 4) bf16 rounding alone can reach
2^-7 = 7.8e-3. binary16 passes with room to spare. That is why the kernels
take binary16 operands."""
import numpy as np
import pytest

from gpu_util import MAX_ABS, REL_L2, errors
from workloads import BY_NAME, prefill_inputs


def round_f16(x):
    return np.asarray(x, np.float32).astype(np.float16).astype(np.float64)


def round_bf16(x):
    """float32 -> nearest bf16 (ties to even), widened to float64."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16 << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def rounded_attention(q, k, v, rnd):
    """Causal GQA attention in fp64 with q, k, v and the weights p rounded by
    rnd; the row sums l use the unrounded p (the kernels sum p in fp32 before
    rounding it for the PV MMA)."""
    n, hq, hd = q.shape
    hkv = k.shape[1]
    g = hq // hkv
    qr, kr, vr = rnd(q), rnd(k), rnd(v)
    scale = 1.0 / np.sqrt(hd)
    mask = np.tril(np.ones((n, n), bool))
    out = np.empty((n, hq, hd))
    for h in range(hq):
        s = (qr[:, h, :] @ kr[:, h // g, :].T) * scale
        s = np.where(mask, s, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        l = p.sum(axis=1, keepdims=True)
        out[:, h, :] = (rnd(p.astype(np.float32)) @ vr[:, h // g, :]) / l
    return out


@pytest.fixture(scope="module")
def case(oracle_mod):
    w = BY_NAME["prefill_f32_n8192_h16x2_d256"]
    n = 512
    q, k, v = prefill_inputs(n, w.n_q_heads, w.n_kv_heads, w.head_dim, w.seed)
    want = oracle_mod.prefill(q, k, v, kv_fmt="f32", sink=0, win=0)
    return q, k, v, want


def test_binary16_operands_meet_the_tolerance(case):
    q, k, v, want = case
    ma, rl = errors(rounded_attention(q, k, v, round_f16), want)
    assert ma <= MAX_ABS and rl <= REL_L2, (ma, rl)
    # with margin: the kernels add fp32 accumulation and exp2 rounding on top
    assert ma <= MAX_ABS / 2 and rl <= REL_L2 / 4, (ma, rl)


def test_bf16_operands_miss_the_tolerance(case):
    q, k, v, want = case
    got = rounded_attention(q, k, v, round_bf16)
    ma, rl = errors(got, want)
    assert ma > MAX_ABS and rl > REL_L2, (ma, rl)
    # the first row alone: v_0 rounded to bf16
    ma0, _ = errors(got[0], want[0])
    assert ma0 > MAX_ABS, ma0


def test_the_rounding_helpers():
    assert round_bf16(np.float32(1.0 + 2 ** -8)) == 1.0            # tie: to even
    assert round_bf16(np.float32(1.0 + 3 * 2 ** -8)) == 1.0 + 2 ** -6  # tie: up to even
    assert round_bf16(np.float32(3.0 + 2 ** -7)) == 3.0             # half-ulp in [2, 4)
    assert round_f16(np.float32(1.0 + 2 ** -11)) == 1.0
    assert round_f16(np.float32(3.0 + 2 ** -9)) == 3.0 + 2 ** -9     # representable
