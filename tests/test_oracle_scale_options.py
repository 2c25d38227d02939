"""Pins of the scale options (blog "[vLLM] Compilation Fusion Passes", section
"Why this design", item 3: E8M0 scales, column-major scales, TMA alignment).

E8M0: every dynamic scale is the smallest power of two not below the plain
scale max(amax / 448, 1e-12) (checked with numpy's frexp, an independent
decomposition), and the codes are the E4M3 values of y / s.  TMA alignment:
the column-major scales are the plain ones at a stride of n rounded up to 4.
"""
import numpy as np
import pytest

import rmsq_inputs as ri

pytestmark = pytest.mark.usefixtures("orc")


def _pow2_ceil(x):
    m, e = np.frexp(x.astype(np.float64))
    return np.where(m == 0.5, x.astype(np.float64), np.ldexp(1.0, e))


@pytest.mark.parametrize("mode", ["fp8_per_token", "fp8_group128_row", "fp8_group64_col"])
def test_e8m0_scales_are_the_next_power_of_two(orc, mode):
    wl = ri.make_workload("e8", 13, 512, res_sigma=1.5, seed=4)
    plain = orc.run_workload(wl, mode, want_y=True)
    e8 = orc.run_workload(wl, mode + "+e8m0")
    s0, s1 = plain["scales"].astype(np.float64), e8["scales"].astype(np.float64)
    assert np.array_equal(s1, _pow2_ceil(plain["scales"]))
    assert np.all(s1 >= s0) and np.all(s1 / 2 < s0)
    # the codes are e4m3(y / s) with the power-of-two scale (an exact scaling)
    y = plain["y"].astype(np.float64)
    n, H = y.shape
    G = H if mode == "fp8_per_token" else (128 if "128" in mode else 64)
    s = s1.reshape(n, 1) if mode == "fp8_per_token" else (s1.T if mode.endswith("_col") else s1)
    v = (y / np.repeat(s, G, axis=1)).astype(np.float32)
    assert np.array_equal(e8["q"], orc.e4m3_encode(v))


def test_e8m0_closed_forms(orc):
    # a row whose amax of y is exactly 448 has plain scale 1, E8M0 scale 1;
    # one with amax 896 has 2 in both; 449 gives a plain scale just above 1
    # and an E8M0 scale of 2
    for amax, want in ((448.0, 1.0), (896.0, 2.0), (449.0, 2.0), (224.0, 0.5)):
        plain = np.float32(max(np.float32(amax) / np.float32(448.0), np.float32(1e-12)))
        assert _pow2_ceil(np.array([plain]))[0] == want


def test_tma_aligned_column_major_stride(orc):
    wl = ri.make_workload("tma", 13, 512, seed=6)   # 13 tokens: stride 16
    plain = orc.run_workload(wl, "fp8_group128_col")
    tma = orc.run_workload(wl, "fp8_group128_col+tma")
    assert tma["scales"].shape == (4, 16)
    assert np.array_equal(tma["scales"][:, :13], plain["scales"])
    assert np.all(tma["scales"][:, 13:] == 0)        # not written
    assert np.array_equal(tma["q"], plain["q"])
    both = orc.run_workload(wl, "fp8_group64_col+e8m0+tma")
    ref = orc.run_workload(wl, "fp8_group64_col+e8m0")
    assert np.array_equal(both["scales"][:, :13], ref["scales"])


@pytest.mark.parametrize("mode", ["fp8_static+e8m0", "nvfp4+e8m0", "fp8_group128_row+tma",
                                  "fp8_per_token+tma"])
def test_options_rejected_where_they_do_not_apply(orc, mode):
    wl = ri.make_workload("bad", 2, 256, seed=1)
    with pytest.raises(RuntimeError):
        orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=1.0)


@pytest.mark.parametrize("mode", ["fp8_per_token", "fp8_group128_row", "fp8_group64_col", "fp8_group128_col"])
def test_ue8m0_bytes_are_the_exponents_of_the_power_of_two_scales(orc, mode):
    """One byte per scale: e such that the E8M0 scale is 2^(e - 127), from
    numpy's frexp of the plain scale (an independent decomposition); the
    codes are those of the power-of-two fp32 scales."""
    wl = ri.make_workload("ue8", 13, 512, res_sigma=1.5, seed=8)
    plain = orc.run_workload(wl, mode)
    pw2 = orc.run_workload(wl, mode + "+e8m0")
    by = orc.run_workload(wl, mode + "+ue8m0")
    assert by["scales"].dtype == np.uint8 and by["scales"].shape == plain["scales"].shape
    m, e = np.frexp(plain["scales"].astype(np.float64))
    want = np.where(m == 0.5, e - 1, e) + 127          # 2^(want - 127) = smallest power of two >= s
    assert np.array_equal(by["scales"].astype(np.int64), want)
    assert np.array_equal(np.ldexp(1.0, by["scales"].astype(np.int64) - 127), pw2["scales"].astype(np.float64))
    assert np.array_equal(by["q"], pw2["q"])


def test_ue8m0_closed_forms_and_tma_stride(orc):
    # an all-zero row: scale floor 1e-12 -> 2^-39 (byte 88); a row whose y
    # amax is just below 448 (inv just below 1) -> scale just below 1 -> 1
    # (byte 127)
    n, H = 2, 128
    x = np.zeros((n, H), np.float64)
    x[1, :] = 1.0
    wl = ri.Workload("z", n, H, "bf16", 1e-6, ri.to_bits(x, "bf16").reshape(n, H), None,
                     ri.to_bits(np.full(H, 448.0), "bf16"))
    r = orc.run_workload(wl, "fp8_per_token+ue8m0")
    assert r["scales"].tolist() == [88, 127]
    wl = ri.make_workload("tma8", 13, 512, seed=9)      # 13 tokens: byte stride 16
    tma = orc.run_workload(wl, "fp8_group128_col+ue8m0+tma")
    ref = orc.run_workload(wl, "fp8_group128_col+ue8m0")
    assert tma["scales"].shape == (4, 16)
    assert np.array_equal(tma["scales"][:, :13], ref["scales"])
    assert np.all(tma["scales"][:, 13:] == 0)
    wl = ri.make_workload("tma8b", 17, 512, seed=9)     # 17 tokens: byte stride 32 (not 20)
    tma = orc.run_workload(wl, "fp8_group64_col+ue8m0+tma")
    ref = orc.run_workload(wl, "fp8_group64_col+ue8m0")
    assert tma["scales"].shape == (8, 32)
    assert np.array_equal(tma["scales"][:, :17], ref["scales"])
    assert np.all(tma["scales"][:, 17:] == 0)


@pytest.mark.parametrize("mode", ["fp8_static+ue8m0", "nvfp4+ue8m0"])
def test_ue8m0_rejected_without_a_dynamic_scale(orc, mode):
    wl = ri.make_workload("bad", 2, 256, seed=1)
    with pytest.raises(RuntimeError):
        orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=1.0)
