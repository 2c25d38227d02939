"""Pins of the oracle's SiLU+Mul + quantisation against the mathematics.

The op (vLLM docs "Fusion torch.compile passes", section "SiLU+Mul +
Quantization (fuse_act_quant)"): a = silu(gate) * up on the gated
up-projection, then the same quantisation as the norm op.  The oracle takes
silu from its plain definition g / (1 + e^-g), evaluated in binary64 and
rounded once; it is pinned here to an extended-precision evaluation on every
bf16 and fp16 input, to closed forms, and the whole op to an independent
double-precision computation plus the quantisation invariants.  A swapped
gate/up, a sign slip in e^-g, a lost factor g or a binary32 evaluation fails
here.
"""
import numpy as np
import pytest

import rmsq_inputs as ri

pytestmark = pytest.mark.usefixtures("orc")


def _ulp_err(got: np.ndarray, want64: np.ndarray) -> np.ndarray:
    """|got - want| in units of the binary32 spacing at want."""
    sp = np.spacing(np.abs(want64).astype(np.float32)).astype(np.float64)
    return np.abs(got.astype(np.float64) - want64) / sp


def _finite_inputs(dtype):
    bits = np.arange(65536, dtype=np.uint32)
    v = (bits << 16).view(np.float32) if dtype == "bf16" else bits.astype(np.uint16).view(np.float16).astype(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_silu_is_the_rounded_definition_on_every_input(orc, dtype):
    """Every finite bf16 / fp16 gate: the oracle's silu equals the binary32
    rounding of g / (1 + e^-g) evaluated in extended precision."""
    g = _finite_inputs(dtype)
    gl = g.astype(np.longdouble)
    want = (gl / (np.longdouble(1) + np.exp(-gl))).astype(np.float32)
    got = orc.silu(g)
    same = (got.view(np.uint32) == want.view(np.uint32))
    assert same.all(), (int((~same).sum()), g[~same][:6].tolist(), got[~same][:6].tolist(), want[~same][:6].tolist())


def test_silu_within_half_an_ulp_of_double(orc):
    rng = np.random.default_rng(7)
    g = np.concatenate([rng.normal(0, 3, 400_000), rng.uniform(-100, 100, 100_000)]).astype(np.float32)
    got = orc.silu(g)
    g64 = g.astype(np.float64)
    want = g64 / (1.0 + np.exp(-g64))
    ok = np.abs(want) > 1e-30
    err = _ulp_err(got[ok], want[ok])
    assert err.max() <= 0.5 + 1e-6, (err.max(), g[ok][np.argmax(err)])


def test_silu_closed_forms(orc):
    s = orc.silu(np.array([0.0, -0.0, 30.0, -120.0, 2.0, -2.0, 1e30, -1e30], np.float32))
    assert s[0] == 0.0 and not np.signbit(s[0])
    assert s[1] == 0.0 and np.signbit(s[1])        # -0 / 2
    assert s[2] == np.float32(30.0)                # e^-30 is below half an ulp of 1
    assert s[3] == 0.0 and np.signbit(s[3])        # -120 / (1 + e^120) underflows to -0
    # silu(x) - silu(-x) = x (each side rounded once)
    assert abs(float(s[4]) - float(s[5]) - 2.0) <= 2 * 2.0 ** -23
    assert s[6] == np.float32(1e30) and s[7] == 0.0 and np.signbit(s[7])


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
    """a = RN32(RN32(silu(g)) * u): the first rounding moves silu by at most
    2^-24 relative, which is less than one ulp of a, and the product's own
    rounding adds half an ulp: within 1.5 ulp of the exact product."""
    wl = ri.make_act_workload("act", 17, 512, dtype=dtype, seed=3)
    r = orc.run_silu_mul(wl.gate_up, mode="fp8_per_token", dtype=dtype, want_y=True)
    want = _act64(wl)
    ok = np.abs(want) > 1e-30
    err = _ulp_err(r["y"][ok], want[ok])
    assert err.max() <= 1.5
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


@pytest.mark.parametrize("mode", ["fp8_static", "fp8_per_token", "fp8_group64_col", "nvfp4",
                                  "fp8_group128_row+e8m0"])
def test_quantisation_of_given_activations(orc, mode):
    """The quantisation step on given fp32 rows is the same step the SiLU+Mul
    op and the norm op end with: fed their own activations it reproduces
    their codes and scales."""
    wl = ri.make_act_workload("act", 11, 512, seed=13)
    scale_in = 0.02 if mode == "fp8_static" else (300.0 if mode == "nvfp4" else 0.0)
    r = orc.run_silu_mul(wl.gate_up, mode=mode, scale_in=scale_in, want_y=True)
    g = orc.run_quant_f32(r["y"], mode=mode, scale_in=scale_in)
    assert np.array_equal(g["q"], r["q"])
    if r["scales"] is not None:
        assert np.array_equal(g["scales"].view(np.uint8), r["scales"].view(np.uint8))
    nw = ri.make_workload("norm", 5, 256, seed=14)
    f = orc.run(nw.x, nw.residual, nw.weight, eps=nw.eps, mode=mode, scale_in=scale_in, want_y=True)
    g = orc.run_quant_f32(f["y"], mode=mode, scale_in=scale_in)
    assert np.array_equal(g["q"], f["q"])
