"""Pins of the oracle's QK-norm + RoPE (vLLM docs "Fusion torch.compile
passes", section "QK Norm + RoPE": split QKV, per-head RMSNorm of Q and K,
rotary embedding).

Position 0 (cos 1, sin 0) reduces every head to the norm op's rounded y; an
independent double-precision normalisation and rotation with the same cos/sin
table agrees to within one step of the activation type; the rotation keeps
each pair's length; v and out-of-range tokens are untouched.  A swapped sin
sign, swapped cos/sin halves, a wrong pair offset or the q weight on k heads
fails one of these.
"""
import numpy as np
import pytest

import rmsq_inputs as ri

pytestmark = pytest.mark.usefixtures("orc")


def _widen(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _ref64(wl):
    """Double-precision normalisation and rotation with the table's fp32 cos/sin."""
    n, D, nh = wl.n_tokens, wl.head_dim, wl.nq + wl.nkv
    x = _widen(wl.qkv[:, :nh * D]).astype(np.float64).reshape(n, nh, D)
    w = np.stack([_widen(wl.q_weight)] * wl.nq + [_widen(wl.k_weight)] * wl.nkv).astype(np.float64)
    y = x / np.sqrt(np.mean(x * x, axis=2, keepdims=True) + wl.eps) * w[None]
    cs = wl.cos_sin[wl.positions].astype(np.float64)
    c, s = cs[:, None, :D // 2], cs[:, None, D // 2:]
    if wl.neox:
        a, b = y[..., :D // 2], y[..., D // 2:]
        out = np.concatenate([a * c - b * s, b * c + a * s], axis=2)
    else:
        a, b = y[..., 0::2], y[..., 1::2]
        out = np.empty_like(y)
        out[..., 0::2], out[..., 1::2] = a * c - b * s, b * c + a * s
    return out.reshape(n, nh * D), y.reshape(n, nh * D)


@pytest.mark.parametrize("neox", [True, False])
def test_against_double_precision(orc, neox):
    wl = ri.make_qk_workload("qk", 23, 8, 2, 128, neox=neox, seed=4)
    got = orc.run_qk_norm_rope(wl)
    nh = wl.nq + wl.nkv
    want64, _ = _ref64(wl)
    g = _widen(got[:, :nh * 128]).astype(np.float64)
    step = np.spacing(np.abs(want64).astype(np.float32)).astype(np.float64) * 2 ** 16   # one bf16 step
    assert np.all(np.abs(g - want64) <= step + 1e-30)
    assert np.mean(got[:, :nh * 128] == ri.to_bits(want64, "bf16").reshape(g.shape)) > 0.98
    assert np.array_equal(got[:, nh * 128:], wl.qkv[:, nh * 128:])          # v untouched


def test_position_zero_is_the_norm_alone(orc):
    wl = ri.make_qk_workload("qk0", 6, 4, 2, 128, seed=7)
    wl.positions[:] = 0
    got = orc.run_qk_norm_rope(wl)
    for h in range(6):
        x = wl.qkv[:, h * 128:(h + 1) * 128]
        w = wl.q_weight if h < 4 else wl.k_weight
        want = orc.run_add_rmsnorm(x, None, w, eps=wl.eps)["y_t"]
        assert np.array_equal(got[:, h * 128:(h + 1) * 128], want), h


def test_rotation_keeps_pair_lengths(orc):
    wl = ri.make_qk_workload("qkl", 16, 4, 2, 128, seed=9)
    got = orc.run_qk_norm_rope(wl)
    _, y64 = _ref64(wl)
    o = _widen(got[:, :6 * 128]).astype(np.float64).reshape(16, 6, 128)
    y = y64.reshape(16, 6, 128)
    lo, lp = o[..., :64] ** 2 + o[..., 64:] ** 2, y[..., :64] ** 2 + y[..., 64:] ** 2
    assert np.allclose(lo, lp, rtol=2 ** -6, atol=1e-6)


def test_out_of_range_positions_leave_the_token_unchanged(orc):
    wl = ri.make_qk_workload("qkr", 5, 4, 2, 128, max_pos=64, seed=3)
    wl.positions[1] = 64
    wl.positions[3] = -1
    got = orc.run_qk_norm_rope(wl)
    assert np.array_equal(got[1], wl.qkv[1]) and np.array_equal(got[3], wl.qkv[3])
    assert not np.array_equal(got[0], wl.qkv[0])


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_quarter_turn_is_an_exact_swap(orc, neox):
    """cos = 0, sin = 1 at every angle: each product is exact (y * 0, y * 1)
    and so is each sum, so a pair (a, b) becomes (-b, a) with no rounding,
    i.e. the norm op's rounded y with the pair swapped and the first element
    negated (compared as values: a zero product may carry either sign)."""
    D = 128
    wl = ri.make_qk_workload("qk90", 7, 4, 2, D, neox=neox, max_pos=8, seed=11)
    wl.positions[:] = 5
    wl.cos_sin[5, :D // 2] = 0.0
    wl.cos_sin[5, D // 2:] = 1.0
    got = orc.run_qk_norm_rope(wl)
    for h in range(6):
        x = wl.qkv[:, h * D:(h + 1) * D]
        w = wl.q_weight if h < 4 else wl.k_weight
        y = _widen(orc.run_add_rmsnorm(x, None, w, eps=wl.eps)["y_t"])
        want = np.empty_like(y)
        if neox:
            want[:, :D // 2], want[:, D // 2:] = -y[:, D // 2:], y[:, :D // 2]
        else:
            want[:, 0::2], want[:, 1::2] = -y[:, 1::2], y[:, 0::2]
        assert np.array_equal(_widen(got[:, h * D:(h + 1) * D]), want), h
