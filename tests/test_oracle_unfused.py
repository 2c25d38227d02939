"""Pins of the unfused two-op sequence (add + RMSNorm writing y in the
activation type, then the quantisation of that tensor).

The first op's y is the fused op's fp32 y rounded to nearest even in the
activation type (rounded here by torch, independently of the oracle); its
residual write-back is the fused op's.  The second op's scales and codes obey
the quantisation invariants on the widened tensor.
"""
import numpy as np
import pytest

import rmsq_inputs as ri

pytestmark = pytest.mark.usefixtures("orc")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("residual", [True, False])
def test_norm_alone_is_rounded_fused_y(orc, dtype, residual):
    wl = ri.make_workload("un", 11, 768, dtype=dtype, residual=residual, res_sigma=1.5, seed=8)
    fused = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token", dtype=dtype, want_y=True)
    un = orc.run_add_rmsnorm(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=dtype)
    want = ri.to_bits(fused["y"].astype(np.float64), dtype).reshape(un["y_t"].shape)
    assert np.array_equal(un["y_t"], want)
    if residual:
        assert np.array_equal(un["residual_out"], fused["residual_out"])
    else:
        assert un["residual_out"] is None


def _widen(bits, dtype):
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    return bits.view(np.float16).astype(np.float32)


@pytest.mark.parametrize("mode", ["fp8_per_token", "fp8_group64_row", "fp8_group128_col+e8m0"])
def test_quant_alone_invariants(orc, mode):
    wl = ri.make_workload("qa", 9, 512, seed=3)
    y_t = orc.run_add_rmsnorm(wl.x, wl.residual, wl.weight, eps=wl.eps)["y_t"]
    r = orc.run_quant(y_t, mode=mode)
    y = _widen(y_t, "bf16").astype(np.float64)
    n, H = y.shape
    base = mode.split("+")[0]
    G = H if base == "fp8_per_token" else (128 if "128" in base else 64)
    sc = r["scales"]
    s = sc.reshape(n, 1) if base == "fp8_per_token" else (sc.T if base.endswith("_col") else sc)
    amax = np.abs(y).reshape(n, H // G, G).max(axis=2)
    plain = np.maximum(amax / 448.0, 1e-12)
    if "e8m0" in mode:
        assert np.all(s >= plain * (1 - 2 ** -23)) and np.all(s / 2 < plain)
    else:
        assert np.allclose(s, plain, rtol=2 ** -23)
    dq = orc.e4m3_decode(r["q"]).astype(np.float64)
    v = y / np.repeat(s.astype(np.float64), G, axis=1)
    e = np.floor(np.log2(np.maximum(np.abs(v), 2.0 ** -6)))
    assert np.all(np.abs(dq - v) <= 0.5 * 2.0 ** (e - 3) * (1 + 2 ** -20) + 1e-30)


def test_unfused_differs_from_fused_only_through_the_rounding(orc):
    """Quantising the widened fp32 y of the fused op with the second op gives
    the fused op's codes exactly when y is representable in T: here every
    |x| = 2 (mean square 4, inv_rms 1/2) and the weights have few significant
    bits, so y = +-w exactly."""
    n, H = 4, 256
    x = ri.to_bits(np.tile(np.array([2.0, -2.0, -2.0, 2.0]), n * H // 4).reshape(n, H), "bf16").reshape(n, H)
    w = ri.to_bits(np.tile(np.array([1.0, 0.5, 0.75, 2.0, 0.25, 3.0, 1.5, 0.125]), H // 8), "bf16")
    fused = orc.run(x, None, w, eps=0.0, mode="fp8_per_token", want_y=True)
    un = orc.run_add_rmsnorm(x, None, w, eps=0.0)
    assert np.array_equal(_widen(un["y_t"], "bf16"), fused["y"])      # y exact in bf16 here
    q = orc.run_quant(un["y_t"], mode="fp8_per_token")
    assert np.array_equal(q["q"], fused["q"]) and np.array_equal(q["scales"], fused["scales"])
