"""Planted mistakes: each mutant is the oracle's C source with one plausible
slip, compiled on the CPU; the pin suite (formats + op pins) must fail on
every one of them.  This is the evidence that the pins hold the oracle to the
pages rather than to itself."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "rmsq_oracle.c")

MUTANTS = [
    ("drop_eps", "sqrtf(ms + a->eps)", "sqrtf(ms)"),
    ("eps_outside_sqrt", "1.0f / sqrtf(ms + a->eps)", "1.0f / (sqrtf(ms) + a->eps)"),
    ("sum_not_mean", "float ms = S / (float)H;", "float ms = S;"),
    ("left_to_right_sum", "float S = oracle_tree_sum_buf(s->sq, H, s->buf);",
     "float S = 0.0f; for (int64_t i = 0; i < H; ++i) S += s->sq[i];"),
    ("no_weight", "(s->h[i] * inv) * widen(a->dtype, a->weight[i])", "(s->h[i] * inv)"),
    ("norm_of_unrounded_sum", "s->h[i] = widen(a->dtype, hb);", "s->h[i] = sum;"),
    ("residual_subtracted", "widen(a->dtype, xr[i]) + widen(a->dtype, a->residual[t * H + i])",
     "widen(a->dtype, xr[i]) - widen(a->dtype, a->residual[t * H + i])"),
    ("times_scale", "oracle_e4m3_encode(y[i] / sc)", "oracle_e4m3_encode(y[i] * sc)"),
    ("scale_over_447", "amax / 448.0f", "amax / 447.0f"),
    ("col_stored_row_major", "store_scale(a, col ? g * a->col_stride + t : t * (H / G) + g, sc);",
     "store_scale(a, t * (H / G) + g, sc);"),
    ("ue8m0_mantissa_byte", "((uint8_t *)a->out_scales)[i] = (uint8_t)((u >> 23) & 0xffu);",
     "((uint8_t *)a->out_scales)[i] = (uint8_t)((u >> 15) & 0xffu);"),
    ("ue8m0_tma_stride_of_4", "const int64_t per16 = (opts & OR_OPT_UE8M0) ? 16 : 4;", "const int64_t per16 = 4;"),
    ("e8m0_rounds_down", "return f == 0.5f ? x : ldexpf(1.0f, k);", "return ldexpf(1.0f, k - 1);"),
    ("tma_stride_not_padded", "*col_stride = (opts & OR_OPT_TMA) ? (n + per16 - 1) / per16 * per16 : n;",
     "*col_stride = n;"),
    # QK-norm + RoPE (pinned by test_oracle_qk.py)
    ("rope_sin_sign", "const float oa = ya * c - yb * s;", "const float oa = ya * c + yb * s;"),
    ("rope_cos_sin_swapped", "const float c = cs[i], s = cs[h + i];", "const float s = cs[i], c = cs[h + i];"),
    ("rope_pair_offset", "b = neox ? i + h : 2 * i + 1;", "b = neox ? (i + h + 1) % (2 * h) : 2 * i + 1;"),
    ("qk_k_heads_use_q_weight", "hd < nq ? q_w : k_w", "q_w"),
    ("group_of_first_half", "for (int k = 0; k < G; ++k) amax = fmaxf(amax, fabsf(yg[k]));",
     "for (int k = 0; k < G / 2; ++k) amax = fmaxf(amax, fabsf(yg[k]));"),
    ("nibbles_swapped", "(uint8_t)(lo | (hi << 4))", "(uint8_t)(hi | (lo << 4))"),
    ("nvfp4_ratio_inverted", "? 0.0f : gs / d;", "? 0.0f : d / gs;"),
    ("nvfp4_block_of_8", "for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(yb[k]));",
     "for (int k = 0; k < 8; ++k) amax = fmaxf(amax, fabsf(yb[k]));"),
    ("nvfp4_over_4", "oracle_e4m3_encode((amax / 6.0f) * gs)", "oracle_e4m3_encode((amax / 4.0f) * gs)"),
    ("e4m3_no_saturation", "if (a >= 448.0f) return (uint8_t)(sign | 0x7e);",
     "if (a >= 480.0f) return (uint8_t)(sign | 0x7f);"),
    ("e4m3_ties_away", "float k = rintf(ldexpf(a, 3 - e));", "float k = floorf(ldexpf(a, 3 - e) + 0.5f);"),
    ("e4m3_bias_8", "int code = ((e + 7) << 3) | ((int)k - 8);", "int code = ((e + 8) << 3) | ((int)k - 8);"),
    ("e2m1_sign_dropped", "uint8_t sign = signbit(v) ? 0x8 : 0x0;", "uint8_t sign = 0;"),
    ("bf16_truncates", "if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1;", ""),
    ("fp16_subnormal_step", "float k = rintf(ldexpf(a, 24));", "float k = rintf(ldexpf(a, 23));"),
    # SiLU+Mul (pinned by test_oracle_act.py)
    ("silu_sign_slip", "gd / (1.0 + exp(-gd))", "gd / (1.0 + exp(gd))"),
    ("silu_sigmoid_only", "gd / (1.0 + exp(-gd))", "1.0 / (1.0 + exp(-gd))"),
    ("silu_without_one", "gd / (1.0 + exp(-gd))", "gd / exp(-gd)"),
    ("silu_in_binary32", "return (float)(gd / (1.0 + exp(-gd)));", "return g / (1.0f + expf(-g));"),
    # all-reduce + RMSNorm (pinned by test_oracle_allreduce.py)
    ("ar_rounds_every_rank", "acc = acc + widen(dtype, partials[(int64_t)r * n * H + i]);",
     "acc = widen(dtype, narrow(dtype, acc + widen(dtype, partials[(int64_t)r * n * H + i])));"),
    ("ar_drops_last_rank", "for (int r = 1; r < nranks; ++r) acc", "for (int r = 1; r < nranks - 1; ++r) acc"),
    ("ar_first_rank_twice", "float acc = widen(dtype, partials[i]);", "float acc = widen(dtype, partials[i]) * 2.0f;"),
    ("gate_up_swapped", "const uint16_t *g = a->x + t * 2 * d, *u = g + d;",
     "const uint16_t *u = a->x + t * 2 * d, *g = u + d;"),
]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pins_catch_planted_mistake(mutant_dir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c_path = mutant_dir / f"{name}.c"
    so_path = mutant_dir / f"lib{name}.so"
    c_path.write_text(mutated)
    subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                           "-shared", "-pthread", str(c_path), "-o", str(so_path), "-lm"])
    env = dict(os.environ, ORACLE_LIB=str(so_path))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(ROOT, "tests", "test_oracle_formats.py"),
                        os.path.join(ROOT, "tests", "test_oracle_op.py"),
                        os.path.join(ROOT, "tests", "test_oracle_act.py"),
                        os.path.join(ROOT, "tests", "test_oracle_scale_options.py"),
                        os.path.join(ROOT, "tests", "test_oracle_qk.py"),
                        os.path.join(ROOT, "tests", "test_oracle_allreduce.py")],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"mutant {name} passed every pin:\n{r.stdout[-2000:]}"
    assert "failed" in r.stdout, r.stdout[-2000:]
