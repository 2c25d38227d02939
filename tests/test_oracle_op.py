"""Pins of the oracle's op against hand-worked rows, closed forms and invariants.

The op (vLLM docs "Fusion torch.compile passes", section "RMSNorm +
Quantization (fuse_norm_quant)"; vLLM PR #51925 summary for NVFP4):
  h = T(x + residual)  (residual updated in place), y = h / rms(h) * w,
  then FP8 E4M3 with a static / per-token / per-group scale, or NVFP4.
Each check below would fail for a plausible slip in the oracle: a dropped
eps, sum instead of mean, a wrong sign or index, y*s instead of y/s, a wrong
constant in the scale, a transposed scale layout, swapped nibbles.
"""
import json
import os

import numpy as np
import pytest
import torch

import rmsq_inputs as ri

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")
FP8_MODES = ["fp8_static", "fp8_per_token", "fp8_group128_row", "fp8_group128_col",
             "fp8_group64_row", "fp8_group64_col"]


def _bits(vals, dtype):
    return ri.to_bits(np.asarray(vals, np.float64), dtype)


def _golden_inputs(ex):
    n, H = ex["n"], ex["H"]

    def fill(v, shape):
        a = np.asarray(v, np.float64)
        return np.broadcast_to(a, shape).copy() if a.size == 1 else a.reshape(shape)

    x = _bits(fill(ex["x"], (n, H)), ex["dtype"]).reshape(n, H)
    r = None if ex["residual"] is None else _bits(fill(ex["residual"], (n, H)), ex["dtype"]).reshape(n, H)
    w = _bits(fill(ex["weight"], (H,)), ex["dtype"])
    return x, r, w


def _expand_hex(h, nbytes):
    b = bytes.fromhex(h)
    return np.frombuffer(b * (nbytes // len(b)) if len(b) < nbytes else b, np.uint8)


def golden_examples():
    return json.load(open(GOLDEN))["examples"]


@pytest.mark.parametrize("ex", golden_examples(), ids=lambda e: e["name"])
def test_golden_worked_examples(orc, ex):
    x, r, w = _golden_inputs(ex)
    out = orc.run(x, r, w, eps=ex["eps"], mode=ex["mode"], scale_in=ex["scale_in"],
                  dtype=ex["dtype"], want_y=True)
    e = ex["expect"]
    q = out["q"].ravel()
    assert np.array_equal(q, _expand_hex(e["q_hex"], q.size))
    if "residual_out_hex" in e:
        ro = out["residual_out"].ravel()
        assert np.all(ro == int(e["residual_out_hex"], 16))
    if "scales_f32_bits" in e:
        s = out["scales"].ravel().view(np.uint32)
        want = [int(v, 16) for v in e["scales_f32_bits"]]
        assert np.all(s == want[0]) if len(want) == 1 else list(s) == want
    if "scales_u8_hex" in e:
        s = out["scales"].ravel()
        want = [int(v, 16) for v in e["scales_u8_hex"]]
        assert np.all(s == want[0]) if len(want) == 1 else list(s) == want
    if "tree_sum" in e:
        h = orc.act_to_float(x[0], ex["dtype"])
        assert orc.tree_sum(h * h) == e["tree_sum"]
        ms = np.uint32(int(e["ms_f32_bits"], 16)).view(np.float32)
        assert np.float32(e["tree_sum"]) / np.float32(ex["H"]) == ms
        inv = np.float32(1) / np.sqrt(ms + np.float32(ex["eps"]))
        assert out["y"][0, 1] == inv     # h = w = 1 there, so y is inv itself


def test_tree_sum_hand_values(orc):
    assert orc.tree_sum([2.0 ** 24, 1, 1, 1]) == 16777218.0     # left-to-right gives 2^24
    assert orc.tree_sum([1, 1, 2.0 ** 24, 1]) == 16777218.0
    assert orc.tree_sum([1.0, 2.0 ** 24, 1.0]) == 16777216.0    # (1 + 2^24) + (1 + 0)
    assert orc.tree_sum([3.0]) == 3.0 and orc.tree_sum([]) == 0.0
    assert orc.tree_sum(np.ones(1000)) == 1000.0


def test_tree_sum_error_bound(orc):
    for n in (7, 64, 1000, 4096, 7168):
        v = (ri.normal(21, n, n) ** 2).astype(np.float32)
        exact = np.sum(v.astype(np.float64))
        P = 1 << (n - 1).bit_length()
        bound = np.log2(P) * 2.0 ** -24 * exact * 1.0001
        assert abs(orc.tree_sum(v) - exact) <= bound


def _small_workloads():
    return [
        ri.make_workload("bf16_res", 24, 512, res_sigma=2.0, eps=1e-5, seed=3),
        ri.make_workload("bf16_nores", 17, 384, residual=False, eps=1e-6, seed=4),
        ri.make_workload("fp16_t3", 9, 1024, dtype="fp16", dist="t3", t_clamp=500.0,
                         n_outliers=8, outlier_mult=50.0, eps=1e-5, seed=5),
        ri.make_workload("bf16_outl", 12, 768, n_outliers=8, outlier_mult=20.0, seed=6),
        # mean square comparable to eps, so that eps visibly changes y
        ri.make_workload("bf16_tiny", 10, 256, x_sigma=1e-3, res_sigma=1e-3, eps=1e-6, seed=7),
    ]


@pytest.mark.parametrize("wl", _small_workloads(), ids=lambda w: w.name)
def test_residual_out_is_rounded_exact_sum(orc, wl):
    if wl.residual is None:
        pytest.skip("no residual")
    out = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token", dtype=wl.dtype)
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    xs = torch.from_numpy(wl.x.view(np.int16)).view(tdt).double()
    rs = torch.from_numpy(wl.residual.view(np.int16)).view(tdt).double()
    want = (xs + rs).float().to(tdt).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out["residual_out"], want)


def _h_f64(orc, wl, out):
    src = out["residual_out"] if wl.residual is not None else wl.x
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float16
    h = torch.from_numpy(np.ascontiguousarray(src).view(np.int16)).view(tdt).double().numpy()
    w = torch.from_numpy(wl.weight.view(np.int16)).view(tdt).double().numpy()
    return h, w


@pytest.mark.parametrize("wl", _small_workloads(), ids=lambda w: w.name)
def test_rms_identity_and_y_closed_form(orc, wl):
    out = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token",
                  dtype=wl.dtype, want_y=True)
    h, w = _h_f64(orc, wl, out)
    y = out["y"].astype(np.float64)
    ms = np.mean(h * h, axis=1)
    # mean((y/w)^2) = ms / (ms + eps)
    lhs = np.mean((y / w) ** 2, axis=1)
    assert np.allclose(lhs, ms / (ms + wl.eps), rtol=1e-5, atol=0)
    # y = h / sqrt(ms + eps) * w up to a few fp32 roundings
    exact = h / np.sqrt(ms + wl.eps)[:, None] * w
    assert np.all(np.abs(y - exact) <= 4 * 2.0 ** -24 * np.abs(exact) + 1e-38)


def _e4m3_step(orc, codes):
    """Distance from |decode(code)| to the next larger E4M3 magnitude."""
    mag = (codes & 0x7f).astype(np.int64)
    table = orc.e4m3_decode(np.arange(0x7f, dtype=np.uint8)).astype(np.float64)
    nxt = np.append(table[1:], 480.0)
    return nxt[np.minimum(mag, 0x7e)] - table[np.minimum(mag, 0x7e)]


def _scales_per_element(mode, scales, n, H):
    if mode == "fp8_per_token":
        return np.repeat(scales[:, None], H, axis=1)
    G = 128 if "128" in mode else 64
    s = scales.T if mode.endswith("_col") else scales
    return np.repeat(s, G, axis=1)


@pytest.mark.parametrize("mode", FP8_MODES)
@pytest.mark.parametrize("wl", _small_workloads(), ids=lambda w: w.name)
def test_fp8_dequant_error_and_amax_code(orc, wl, mode):
    if "group128" in mode and wl.hidden % 128:
        pytest.skip("hidden not a multiple of 128")
    s_in = 0.05 if mode == "fp8_static" else 0.0
    out = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=s_in,
                  dtype=wl.dtype, want_y=True)
    y, q = out["y"].astype(np.float64), out["q"]
    n, H = y.shape
    if mode == "fp8_static":
        s = np.full_like(y, np.float32(s_in))
    else:
        s = _scales_per_element(mode, out["scales"], n, H).astype(np.float64)
    deq = orc.e4m3_decode(q).astype(np.float64)
    ratio = y / s
    unsat = np.abs(ratio) <= 448.0
    err = np.abs(deq - ratio)
    half_step = 0.5 * _e4m3_step(orc, q)
    assert np.all(err[unsat] <= half_step[unsat] * (1 + 2.0 ** -20) + np.abs(ratio[unsat]) * 2.0 ** -23)
    assert np.all(np.sign(deq[deq != 0]) == np.sign(ratio[deq != 0]))
    if mode != "fp8_static":
        # every element fits: |y| <= 448 s (up to the fp32 rounding of amax/448) ...
        assert np.all(np.abs(ratio) <= 448.0 * (1 + 2.0 ** -22))
        # ... and the largest magnitude of each scale unit lands on the top code 448
        mags = (q & 0x7f).reshape(n, -1, 64 if "64" in mode else (128 if "128" in mode else H))
        assert np.all(mags.max(axis=2) == 0x7e)


def test_group_col_is_transpose_of_row(orc):
    wl = ri.make_workload("t", 10, 512, seed=8)
    for G in (128, 64):
        a = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=f"fp8_group{G}_row")
        b = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=f"fp8_group{G}_col")
        assert np.array_equal(a["q"], b["q"])
        assert a["scales"].shape == (10, 512 // G) and b["scales"].shape == (512 // G, 10)
        assert np.array_equal(a["scales"].T, b["scales"])


@pytest.mark.parametrize("wl", _small_workloads(), ids=lambda w: w.name)
def test_nvfp4_invariants(orc, wl):
    out = orc.run_workload(wl, "nvfp4", want_y=True)
    gs = np.float64(out["scale_in"])
    y = out["y"].astype(np.float64)
    n, H = y.shape
    assert np.isclose(gs * np.abs(y).max(), 2688.0, rtol=2.0 ** -22)
    sb = out["scales"]
    d = orc.e4m3_decode(sb).astype(np.float64)                      # [n, H/16]
    amax = np.abs(y).reshape(n, H // 16, 16).max(axis=2)
    ideal = amax / 6.0 * gs
    normal = ideal >= 2.0 ** -6
    # block scale is the E4M3 rounding of amax/6 * gs: within half a step (relative 2^-4)
    assert np.all(np.abs(d - ideal)[normal] <= ideal[normal] * 2.0 ** -4 * 1.0001)
    assert np.all(d <= 448.0)
    # unpack nibbles: element 2j is the low nibble of byte j
    lo, hi = out["q"] & 0xF, out["q"] >> 4
    codes = np.empty((n, H), np.uint8)
    codes[:, 0::2], codes[:, 1::2] = lo, hi
    deq = orc.e2m1_decode(codes).astype(np.float64)
    r = np.where(d == 0, 0.0, gs / np.where(d == 0, 1, d))
    yr = y * np.repeat(r, 16, axis=1)
    unsat = np.abs(yr) <= 6.0
    steps = np.array([0.5, 0.5, 0.5, 0.5, 1, 1, 2, 2], np.float64)[codes & 7]
    assert np.all(np.abs(deq - yr)[unsat] <= 0.5 * steps[unsat] * (1 + 2.0 ** -20) + 1e-30)
    # the largest element of each block with a normal scale lands on the top code 6
    top = (codes & 7).reshape(n, H // 16, 16).max(axis=2)
    assert np.all(top[normal] == 7)


def test_thread_count_does_not_change_results(orc):
    wl = ri.make_workload("t", 33, 1024, res_sigma=2.0, seed=9)
    for mode in ("fp8_per_token", "fp8_group128_col", "nvfp4"):
        a = orc.run(wl.x, wl.residual, wl.weight, eps=1e-5, mode=mode, scale_in=100.0)
        b = orc.run(wl.x, wl.residual, wl.weight, eps=1e-5, mode=mode, scale_in=100.0, nthreads=5)
        for k in ("q", "scales", "residual_out"):
            assert np.array_equal(a[k], b[k])


def test_static_scale_direction(orc):
    """Doubling the static scale halves every unsaturated y/s: codes shift down by
    exactly one binade (8 codes) for normal values."""
    wl = ri.make_workload("t", 4, 256, seed=10)
    a = orc.run(wl.x, wl.residual, wl.weight, eps=1e-6, mode="fp8_static", scale_in=0.01, want_y=True)
    b = orc.run(wl.x, wl.residual, wl.weight, eps=1e-6, mode="fp8_static", scale_in=0.02)
    ratio = np.abs(a["y"] / np.float32(0.01))
    ok = (ratio >= 2.0 ** -5) & (ratio <= 440.0)
    assert np.all((a["q"] & 0x7f)[ok].astype(int) - (b["q"] & 0x7f)[ok].astype(int) == 8)


# ------------------------------------------------------------------ NVFP4 with a data-derived global scale
def test_nvfp4_dynamic_all_twos_row(orc):
    """All-twos row: y = 1 everywhere, so amax = 1 and gs = 2688 = 0x45280000;
    then exactly the hand-worked static row: block scale 0x7E, bytes 0x77."""
    x = ri.to_bits(np.ones((3, 32)), "bf16").reshape(3, 32)
    w = ri.to_bits(np.ones(32), "bf16")
    out = orc.run_nvfp4_dynamic(x, x, w, eps=0.0)
    assert out["global_scale"].view(np.uint32)[0] == 0x45280000
    assert np.all(out["q"] == 0x77) and np.all(out["scales"] == 0x7E)
    assert np.all(out["residual_out"] == 0x4000)


def test_nvfp4_dynamic_all_zero_batch(orc):
    """amax = 0: the global scale falls back to 1 and every code is +0."""
    x = np.zeros((2, 64), np.uint16)
    w = ri.to_bits(np.ones(64), "bf16")
    out = orc.run_nvfp4_dynamic(x, None, w, eps=1e-6)
    assert out["global_scale"][0] == 1.0
    assert not out["q"].any() and not out["scales"].any()


@pytest.mark.parametrize("wl", _small_workloads(), ids=lambda w: w.name)
def test_nvfp4_dynamic_matches_static_with_batch_amax(orc, wl):
    if wl.hidden % 16:
        pytest.skip("hidden not a multiple of 16")
    dyn = orc.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=wl.dtype)
    pre = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token",
                  dtype=wl.dtype, want_y=True)
    amax = np.float32(np.abs(pre["y"]).max())
    assert dyn["global_scale"][0] == np.float32(2688.0) / amax
    assert abs(float(dyn["global_scale"][0]) * float(amax) - 2688.0) <= 2688.0 * 2.0 ** -23
    st = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode="nvfp4",
                 scale_in=float(dyn["global_scale"][0]), dtype=wl.dtype)
    for k in ("q", "scales", "residual_out"):
        assert np.array_equal(dyn[k], st[k]) if st[k] is not None else dyn[k] is None
