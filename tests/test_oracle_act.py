"""Pins of the oracle's SiLU+Mul + quantisation against the mathematics.

The op (vLLM docs "Fusion torch.compile passes", section "SiLU+Mul +
Quantization (fuse_act_quant)"): a = silu(gate) * up on the gated
up-projection, then the same quantisation as the norm op.  The oracle's e^x
(Cody-Waite reduction, degree-7 Taylor polynomial) is pinned against the
double-precision exponential of numpy, silu against its double-precision
definition, and the whole op against an independent double-precision
computation plus the quantisation invariants.  A swapped gate/up, a sign slip
in e^-g, a missing term of the polynomial or a wrong ln2 split fails here.
"""
import math

import numpy as np
import pytest

import rmsq_inputs as ri

pytestmark = pytest.mark.usefixtures("orc")


def _ulp_err(got: np.ndarray, want64: np.ndarray) -> np.ndarray:
    """|got - want| in units of the binary32 spacing at want."""
    sp = np.spacing(np.abs(want64).astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - want64) / sp


def test_exp_accuracy_over_the_normal_range(orc):
    x = np.concatenate([np.linspace(-87.3, 88.7, 1_500_001), np.linspace(-1, 1, 200_001)]).astype(np.float32)
    got = orc.expf(x)
    want = np.exp(x.astype(np.float64))
    err = _ulp_err(got, want)
    assert err.max() <= 2.0, (err.max(), x[np.argmax(err)])
    assert np.mean(err) < 0.6


def test_exp_special_values(orc):
    e = orc.expf(np.array([0.0, -0.0, 1.0, 89.5, 200.0, -105.0, -1e30, np.inf, -np.inf, np.nan], np.float32))
    assert e[0] == 1.0 and e[1] == 1.0
    assert e[2] == np.float32(math.e)            # the binary32 nearest to e
    assert np.isinf(e[3]) and np.isinf(e[4]) and e[3] > 0
    assert e[5] == 0.0 and e[6] == 0.0 and e[8] == 0.0
    assert np.isinf(e[7])
    assert np.isnan(e[9])


def test_exp_overflow_and_subnormal_edges(orc):
    # largest x with a finite e^x, and the subnormal range (absolute error
    # below one subnormal step there)
    x_hi = np.float32(88.72283)
    assert np.isfinite(orc.expf(np.array([x_hi], np.float32)))[0]
    assert np.isinf(orc.expf(np.array([88.73], np.float32)))[0]
    x = np.linspace(-103.9, -87.4, 100_001).astype(np.float32)
    got = orc.expf(x).astype(np.float64)
    want = np.exp(x.astype(np.float64))
    tiny = 2.0 ** -149
    assert np.max(np.abs(got - want) - 2 * np.spacing(want.astype(np.float32)).astype(np.float64)) <= tiny


def test_silu_against_its_definition(orc):
    rng = np.random.default_rng(7)
    g = np.concatenate([rng.normal(0, 3, 400_000), rng.uniform(-100, 100, 100_000)]).astype(np.float32)
    got = orc.silu(g)
    g64 = g.astype(np.float64)
    want = g64 / (1.0 + np.exp(-g64))
    ok = np.abs(want) > 1e-30
    err = _ulp_err(got[ok], want[ok])
    assert err.max() <= 3.0, (err.max(), g[ok][np.argmax(err)])


def test_silu_closed_forms(orc):
    s = orc.silu(np.array([0.0, 30.0, -120.0, 2.0, -2.0], np.float32))
    assert s[0] == 0.0
    assert s[1] == np.float32(30.0)                # e^-30 below half an ulp of 1
    assert s[2] == 0.0 and np.signbit(s[2])        # -120 / inf = -0
    # silu(x) - silu(-x) = x
    assert abs(float(s[3]) - float(s[4]) - 2.0) < 4e-7


def _act64(wl):
    gu = wl.gate_up
    d = wl.d
    tof = (lambda b: (b.astype(np.uint32) << 16).view(np.float32)) if wl.dtype == "bf16" else \
        (lambda b: b.view(np.float16).astype(np.float32))
    g = tof(gu[:, :d]).astype(np.float64)
    u = tof(gu[:, d:]).astype(np.float64)
    return g / (1.0 + np.exp(-g)) * u


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_activation_matches_double_precision(orc, dtype):
    wl = ri.make_act_workload("act", 17, 512, dtype=dtype, seed=3)
    r = orc.run_silu_mul(wl.gate_up, mode="fp8_per_token", dtype=dtype, want_y=True)
    want = _act64(wl)
    ok = np.abs(want) > 1e-30
    err = _ulp_err(r["y"][ok], want[ok])
    assert err.max() <= 5.0
    # gate and up are not interchangeable: the swapped product is far off
    d = wl.d
    swapped = ri.ActWorkload("sw", wl.n_tokens, d, dtype,
                             np.concatenate([wl.gate_up[:, d:], wl.gate_up[:, :d]], axis=1))
    r2 = orc.run_silu_mul(swapped.gate_up, mode="fp8_per_token", dtype=dtype, want_y=True)
    assert np.max(np.abs(r2["y"] - want)) > 0.1


@pytest.mark.parametrize("mode", ["fp8_per_token", "fp8_group128_row", "fp8_group64_col"])
def test_dynamic_scales_and_dequant_bound(orc, mode):
    wl = ri.make_act_workload("act", 9, 1024, seed=11)
    r = orc.run_silu_mul(wl.gate_up, mode=mode, want_y=True)
    y, q, sc = r["y"].astype(np.float64), r["q"], r["scales"]
    n, d = y.shape
    G = d if mode == "fp8_per_token" else (128 if "128" in mode else 64)
    s = sc.reshape(n, 1) if mode == "fp8_per_token" else (sc.T if mode.endswith("_col") else sc)
    s = np.repeat(s.astype(np.float64), G, axis=1)
    # scale = amax / 448 per unit (floored at 1e-12)
    amax = np.abs(y).reshape(n, d // G, G).max(axis=2)
    assert np.allclose(s[:, ::G], np.maximum(amax / 448.0, 1e-12), rtol=2 ** -23)
    dq = orc.e4m3_decode(q).astype(np.float64)
    v = y / s
    # half an E4M3 step at |v| (step 2^(e-3) for normals, 2^-9 below 2^-6)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
    half = 0.5 * 2.0 ** (e - 3)
    assert np.all(np.abs(dq - v) <= half * (1 + 2 ** -20) + 1e-30)
    # every unit reaches the top code 448 (0x7e) in magnitude
    top = np.abs(dq).reshape(n, d // G, G).max(axis=2)
    assert np.all(top == 448.0)


def test_nvfp4_block_scales(orc):
    wl = ri.make_act_workload("act", 6, 256, seed=5)
    r = orc.run_silu_mul_workload(wl, "nvfp4", want_y=True)
    y, sc, gs = r["y"].astype(np.float64), r["scales"], np.float32(r["scale_in"])
    d = orc.e4m3_decode(sc).astype(np.float64)
    amax = np.abs(y).reshape(6, 16, 16).max(axis=2)
    # the block scale is the E4M3 value nearest (amax / 6) * gs, within half a step
    tgt = (amax / 6.0) * float(gs)
    e = np.floor(np.log2(np.maximum(tgt, 2.0 ** -6)))
    assert np.all(np.abs(d - np.minimum(tgt, 448.0)) <= 0.5 * 2.0 ** (e - 3) * (1 + 2 ** -20))
    assert np.max(d) == 448.0      # gs = 2688 / amax puts the largest block at the top code
