"""Pins of the oracle's all-reduce + residual add + RMSNorm + quantisation
(vLLM docs "Fusion torch.compile passes", section "AllReduce + RMSNorm
(fuse_allreduce_rms)"; reading R22: the ranks' partial tensors summed in rank
order in binary32, rounded once to the activation type, then the fused op).

Pinned to the fused op itself (one rank, a zero partner rank, an exactly
doubled activation, cancelling ranks), to the exact sum rounded once where
binary32 holds it exactly, and to a closed form where rounding after every
rank would give another result.
"""
import numpy as np
import pytest
import torch

import rmsq_inputs as ri

pytestmark = pytest.mark.usefixtures("orc")
MODES = ["fp8_static", "fp8_per_token", "fp8_group64_col", "nvfp4", "fp8_group128_row+ue8m0"]


def _same(a, b):
    for k in ("q", "scales", "residual_out"):
        if a[k] is None:
            assert b[k] is None
        else:
            assert np.array_equal(a[k].view(np.uint8), b[k].view(np.uint8)), k


def _scale(mode):
    return 0.05 if mode == "fp8_static" else (400.0 if mode == "nvfp4" else 0.0)


@pytest.mark.parametrize("mode", MODES)
def test_one_rank_and_a_zero_rank_are_the_fused_op(orc, mode):
    wl = ri.make_workload("ar1", 9, 512, res_sigma=1.5, seed=71)
    ref = orc.run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=_scale(mode))
    one = orc.run_allreduce(wl.x[None], wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=_scale(mode))
    _same(one, ref)
    zero = np.zeros_like(wl.x)
    for parts in ((wl.x, zero), (zero, wl.x, zero)):
        r = orc.run_allreduce(np.stack(parts), wl.residual, wl.weight, eps=wl.eps, mode=mode,
                              scale_in=_scale(mode))
        _same(r, ref)


def test_two_equal_ranks_double_the_activation(orc):
    wl = ri.make_workload("ar2", 7, 1024, residual=False, seed=72)
    xf = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).float().numpy()
    doubled = ri.to_bits(2.0 * xf.astype(np.float64), "bf16").reshape(wl.x.shape)    # exact in bf16
    ref = orc.run(doubled, None, wl.weight, eps=wl.eps, mode="fp8_per_token")
    r = orc.run_allreduce(np.stack([wl.x, wl.x]), None, wl.weight, eps=wl.eps, mode="fp8_per_token")
    _same(r, ref)


def test_cancelling_ranks_leave_the_residual(orc):
    wl = ri.make_workload("ar3", 5, 256, res_sigma=1.0, seed=73)
    neg = wl.x ^ np.uint16(0x8000)                       # -x, exactly
    r = orc.run_allreduce(np.stack([wl.x, neg]), wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token")
    assert np.array_equal(r["residual_out"], wl.residual)   # h = T(0 + r) = r


@pytest.mark.parametrize("R", [2, 3, 8])
def test_reduced_activation_is_the_exact_sum_rounded_once(orc, R):
    """With a zero residual, residual_out is the reduced activation itself.
    Seeded partials whose binary32 sums are exact: it equals the exact
    (binary64) sum rounded once to bf16."""
    n, H = 6, 512
    parts = np.stack([ri.to_bits(ri.normal(80 + r, 1, n * H), "bf16").reshape(n, H) for r in range(R)])
    vals = torch.from_numpy(parts.view(np.int16)).view(torch.bfloat16).double().numpy()
    exact = vals.sum(axis=0)
    f32 = vals.astype(np.float32)
    seq = f32[0].copy()
    for r in range(1, R):
        seq = seq + f32[r]
    exact_ok = seq.astype(np.float64) == exact
    assert exact_ok.mean() > 0.999
    w = ri.to_bits(np.ones(H), "bf16")
    out = orc.run_allreduce(parts, np.zeros((n, H), np.uint16), w, eps=1e-6, mode="fp8_per_token")
    want = ri.to_bits(exact, "bf16").reshape(n, H)
    assert np.array_equal(out["residual_out"][exact_ok], want[exact_ok])


def test_sum_rounds_once_not_after_every_rank(orc):
    """1 + 2^-9 + 2^-9 + 2^-9 = 1 + 0.75 * 2^-7: rounded once to bf16 it is
    1 + 2^-7 (0x3F81); rounding after every addition would stay at 1 (0x3F80)."""
    H = 16
    parts = np.stack([ri.to_bits(np.full((1, H), v), "bf16").reshape(1, H) for v in (1.0, 2.0 ** -9, 2.0 ** -9,
                                                                                  2.0 ** -9)])
    out = orc.run_allreduce(parts, np.zeros((1, H), np.uint16), ri.to_bits(np.ones(H), "bf16"), eps=1e-6,
                            mode="fp8_static", scale_in=1.0)
    assert np.all(out["residual_out"] == 0x3F81)
