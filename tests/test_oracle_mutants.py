"""The oracle's pins can fail: plant one plausible mistake at a time in a copy
of the oracle, on the CPU, and check that test_oracle_pins.py rejects it.

Each mutant replaces one exact piece of oracle/oracle.c or oracle/oracle.py
(the piece must occur exactly once) in a copy of the package under a temporary
directory; the pins then run in a child pytest with FA_ORACLE_MUTANT_DIR
pointing there (conftest.py puts it first on sys.path). A mutant the pins pass
is a gap in the pins. The real oracle is never modified.
"""
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, file, exact text, replacement): each a mistake a restatement of the
# pages could plausibly make.
# Left out because they are equivalent to the oracle (no input tells them
# apart): dropping the id = 0 guard of an all-zero Q4_0 block (0 * inf is NaN,
# whose code is 0 + 8, the same code) and dropping the shadow_win > 0 test of the
# read rule (with shadow_win 0, s > p - 0 never holds for a key s <= p).
MUTANTS = [
    # binary16 conversion
    ("f16_ties_away", "oracle.c", "(rem == 0x1000u && (h & 1u))", "(rem == 0x1000u)"),
    ("f16_subnormal_shift", "oracle.c", "const int s = -(E + 1); /* >= 14 */",
     "const int s = -E; /* >= 14 */"),
    # fp8 e4m3fn
    ("e4m3_saturates_late", "oracle.c", "(e == 8 && q > 14.0)", "(e == 8 && q > 15.0)"),
    ("e4m3_subnormal_bound", "oracle.c", "if (e < -6) {", "if (e < -7) {"),
    ("e4m3_ties_up", "oracle.c",
     "if (r > 0.5 || (r == 0.5 && fmod(q, 2.0) == 1.0))\n        q += 1.0;\n    if (q == 16.0)",
     "if (r >= 0.5)\n        q += 1.0;\n    if (q == 16.0)"),
    ("e4m3_store_multiplies", "oracle.c", "const float t = x[i] / scale;",
     "const float t = x[i] * scale;"),
    ("e4m3_load_divides", "oracle.c", "const float w = v * scale;", "const float w = v / scale;"),
    # Q4_0 blocks
    ("q4_scale_positive", "oracle.c", "const float d = amax / -8.0f;",
     "const float d = amax / 8.0f;"),
    ("q4_offset_7", "oracle.c", "(int32_t)((uint32_t)qv + 8u)", "(int32_t)((uint32_t)qv + 7u)"),
    ("q4_nibbles_swapped", "oracle.c",
     "(oracle_q4_code(t_lo) | (oracle_q4_code(t_hi) << 4))",
     "(oracle_q4_code(t_hi) | (oracle_q4_code(t_lo) << 4))"),
    ("q4_decode_offset", "oracle.c", "out[j] = (double)((b[2 + j] & 0xf) - 8) * d;",
     "out[j] = (double)((b[2 + j] & 0xf) - 7) * d;"),
    ("q4_rni_ties_odd", "oracle.c", "(frac == 0.5 && fmod(r, 2.0) != 0.0)",
     "(frac == 0.5 && fmod(r, 2.0) == 0.0)"),
    ("q4_amax_signed", "oracle.c", "amax = fmaxf(amax, fabsf(x[j]));",
     "amax = fmaxf(amax, x[j]);"),
    # attended set
    ("window_one_wider", "oracle.c", "(j >= p - win + 1)", "(j >= p - win)"),
    ("sink_one_more", "oracle.c", "return (j < sink) ||", "return (j <= sink) ||"),
    ("no_diagonal", "oracle.c", "if (j < 0 || j > p)", "if (j < 0 || j >= p)"),
    ("win0_means_empty_window", "oracle.c", "if (win <= 0)\n        return 1;",
     "if (win < 0)\n        return 1;"),
    ("tile_map_short_tile", "oracle.c", "j < L && j < kt * bk + bk; j++)",
     "j < L && j < kt * bk + bk - 1; j++)"),
    # which copy a Q4_0 reader sees
    ("shadow_window_one_wider", "oracle.c", "s > p - shadow_win &&", "s >= p - shadow_win &&"),
    ("ring_floor_one_lower", "oracle.c", "s > L - 1 - ORACLE_RING_ROWS",
     "s >= L - 1 - ORACLE_RING_ROWS"),
    ("no_ring_floor", "oracle.c", "s > p - shadow_win && s > L - 1 - ORACLE_RING_ROWS",
     "s > p - shadow_win"),
    ("shadow_sink_one_more", "oracle.c", "if (s < shadow_sink)", "if (s <= shadow_sink)"),
    # attention arithmetic
    ("gqa_head_modulo", "oracle.c", "const int g = h / G; /* [B]",
     "const int g = h % Hkv; /* [B]"),
    ("no_score_scale", "oracle.c", "sc[j] = scale * dot;", "sc[j] = dot;"),
    ("den_squares_weights", "oracle.c", "den += w;\n", "den += w * w;\n"),
    ("lse_without_max", "oracle.c", "lse[rh] = m + log(den);", "lse[rh] = log(den);"),
    ("v_reads_key_row", "oracle.c",
     "const double *vr = oracle_key_row(vbody, vf16, p, j, g, L, Hkv, hd, shadow_sink,\n"
     "                                              shadow_win);",
     "const double *vr = oracle_key_row(kbody, kf16, p, j, g, L, Hkv, hd, shadow_sink,\n"
     "                                              shadow_win);"),
    # MergeAttnStates
    ("merge_weights_swapped", "oracle.c",
     "prefix[row + d] * (wp / tot) + suffix[row + d] * (ws / tot)",
     "prefix[row + d] * (ws / tot) + suffix[row + d] * (wp / tot)"),
    ("merge_context_off_by_one", "oracle.c", "with_context >= 0 && t >= with_context",
     "with_context >= 0 && t > with_context"),
    ("merge_lse_without_max", "oracle.c", "out_lse[li] = log(tot) + m;",
     "out_lse[li] = log(tot);"),
    ("merge_pos_inf_kept", "oracle.c", "if (lp == INFINITY)\n                lp = -INFINITY;",
     "if (lp == INFINITY)\n                lp = INFINITY;"),
    # split-KV decode
    ("plan_no_round_to_16", "oracle.c", "split_len = (split_len + 15) / 16 * 16;",
     "split_len = split_len;"),
    ("partial_unscaled_weight", "oracle.c", "const double w = exp(scale * dot - m);",
     "const double w = exp(dot - m);"),
    ("partial_gqa_modulo", "oracle.c", "const int g = h / G;\n        const float *qr = q + (int64_t)h * hd;",
     "const int g = h % Hkv;\n        const float *qr = q + (int64_t)h * hd;"),
    ("combine_no_rescale_of_l", "oracle.c", "den += w * l[s];", "den += l[s];"),
    ("combine_inverted_weight", "oracle.c", "const double w = exp(m[s] - M);",
     "const double w = exp(M - m[s]);"),
    # edge branches
    ("f16_overflow_not_inf", "oracle.c", "    if (E > 15)\n        return (uint16_t)(sign | 0x7c00u);",
     "    if (E > 15)\n        return (uint16_t)(sign | 0x7bffu);"),
    ("f16_nan_becomes_inf", "oracle.c", "(man ? 0x7e00u : 0x7c00u)", "(0x7c00u)"),
    ("e4m3_nan_saturates", "oracle.c", "    if (isnan(f))\n        return 0x7f;",
     "    if (isnan(f))\n        return 0x7e;"),
    ("e4m3_neg_zero_positive", "oracle.c", "    if (a == 0.0)\n        return sign;",
     "    if (a == 0.0)\n        return 0;"),
    ("q4_no_low_clamp", "oracle.c", "    if (c < 0)\n        return 0;", "    if (c < 0)\n        return c & 15;"),
    ("q4_no_high_clamp", "oracle.c", "    if (c > 15)\n        return 15;", "    if (c > 15)\n        return c & 15;"),
    ("q4_nan_not_zero", "oracle.c", "    if (isnan(t))\n        return 0;", "    if (isnan(t))\n        return 7;"),
    ("tile_map_ignores_offset", "oracle.c", "if (oracle_visible(pos0 + t, j, sink, win))",
     "if (oracle_visible(t, j, sink, win))"),
    ("partial_empty_not_zeroed", "oracle.c", "        for (int e = 0; e < hd; e++)\n            acc[e] = 0.0;",
     "        for (int e = 1; e < hd; e++)\n            acc[e] = 0.0;"),
    ("combine_all_empty_ok", "oracle.c", "    if (M == -INFINITY)\n        return -1;",
     "    if (M == -INFINITY)\n        return 0;"),
    ("merge_both_empty_takes_suffix", "oracle.c",
     "                for (int d = 0; d < D; d++)\n                    out[row + d] = prefix[row + d];\n                out_lse[li] = -INFINITY;",
     "                for (int d = 0; d < D; d++)\n                    out[row + d] = suffix[row + d];\n                out_lse[li] = -INFINITY;"),
    ("attention_sees_only_window", "oracle.c", "return (j < sink) || (j >= p - win + 1);",
     "return (j >= p - win + 1);"),
    ("q4_high_saturation_zero", "oracle.c", "    if (td >= 2147483648.0)\n        return INT32_MAX;",
     "    if (td >= 2147483648.0)\n        return 0;"),
    ("q4_offset_saturates", "oracle.c", "(int32_t)((uint32_t)qv + 8u)",
     "(qv > 2147483639 ? 2147483647 : qv + 8)"),
    ("plan_cap_ignored", "oracle.c", "    if (ns > cap)\n        ns = cap;", "    (void)cap;"),
    ("merge_suffix_pos_inf_kept", "oracle.c", "if (ls == INFINITY)\n                ls = -INFINITY;",
     "if (ls == INFINITY)\n                ls = INFINITY;"),
    ("partial_max_not_subtracted", "oracle.c", "const double w = exp(scale * dot - m);",
     "const double w = exp(scale * dot);"),
    # the numpy front end
    ("chunk_offset_dropped", "oracle.py", "return attention(q[rows], rows + pos0, kk, vv,",
     "return attention(q[rows], rows, kk, vv,"),
    ("q4_shadow_copy_dropped", "oracle.py", "self.f16 = f16_to_f64(f16_rne(x_f32))",
     "self.f16 = None"),
    ("v_scale_from_k", "oracle.py", "KVValues(v[:L], kv_fmt, v_scale)",
     "KVValues(v[:L], kv_fmt, k_scale)"),
]


def _make_mutant(tmp, name, fname, old, new):
    pkg = os.path.join(tmp, name, "oracle")
    shutil.copytree(ORACLE, pkg, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    path = os.path.join(pkg, fname)
    with open(path) as f:
        src = f.read()
    assert src.count(old) == 1, f"{name}: the mutated text must occur once in {fname}"
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return os.path.dirname(pkg)


def _run_pins(mutant_dir):
    # The mutant must build: a compile error would fail the pins for the wrong
    # reason.
    b = subprocess.run([sys.executable, "-c", "from oracle import build; build.build()"],
                       cwd=mutant_dir, capture_output=True, text=True)
    if b.returncode != 0:
        return 100 + b.returncode, "the mutant did not build:\n" + b.stderr[-2000:]
    env = dict(os.environ, FA_ORACLE_MUTANT_DIR=mutant_dir, OMP_NUM_THREADS="2")
    r = subprocess.run([sys.executable, "-m", "pytest", PINS, "-x", "-q", "-p",
                        "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True)
    return r.returncode, r.stdout[-2000:] + r.stderr[-2000:]


def test_mutant_texts_are_unique():
    for name, fname, old, new in MUTANTS:
        with open(os.path.join(ORACLE, fname)) as f:
            assert f.read().count(old) == 1, name
        assert old != new, name


def test_pins_reject_every_mutant(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc is needed to build the mutant oracles")
    dirs = {m[0]: _make_mutant(str(tmp_path), *m) for m in MUTANTS}
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        results = dict(zip(dirs, ex.map(_run_pins, dirs.values())))
    survivors = {n: out for n, (rc, out) in results.items() if rc != 1}
    # rc 1 is "some test failed"; anything else (0 = all passed, 2+ = the run
    # itself broke) leaves the mutant unkilled.
    assert not survivors, "mutants the pins did not reject:\n" + "\n".join(
        f"--- {n} (rc={results[n][0]})\n{out}" for n, out in survivors.items())


def test_pins_pass_on_an_unmodified_copy(tmp_path):
    pkg = os.path.join(str(tmp_path), "oracle")
    shutil.copytree(ORACLE, pkg, ignore=shutil.ignore_patterns("_build", "__pycache__"))
    rc, out = _run_pins(str(tmp_path))
    assert rc == 0, out
