"""Scale options on the GPU (E8M0 power-of-two scales, TMA-aligned
column-major stride) against the oracle, bit for bit, for the norm op in every
kernel variant and for SiLU+Mul; padding entries of the aligned layout are not
written."""
import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu
OPTION_MODES = ["fp8_per_token+e8m0", "fp8_group128_row+e8m0", "fp8_group64_col+e8m0",
                "fp8_group128_col+tma", "fp8_group64_col+e8m0+tma"]
SENTINEL = 0x7f7f7f7f


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def _scales_out(mode, n, H):
    sc = rq.scales_like(mode, n, H, "cuda")
    sc.view(torch.int32).fill_(SENTINEL)
    return sc


def _check_scales(got_sc, want_sc, mode, n, label):
    g = got_sc.cpu().numpy()
    if "+tma" in mode:
        assert np.all(g[:, n:].view(np.int32) == SENTINEL), f"{label}: padding written"
        g, want_sc = g[:, :n], want_sc[:, :n]
    assert np.array_equal(g.view(np.uint32), want_sc.view(np.uint32)), f"{label}: scales differ"


@pytest.mark.parametrize("mode", OPTION_MODES)
@pytest.mark.parametrize("n", [13, 900])
def test_norm_op_with_options(mode, n):
    wl = ri.make_workload(f"opt_{n}", n, 1024, res_sigma=1.5, seed=n)
    want = oracle.run_workload(wl, mode)
    x, r, w = (P.dev_act(a, wl.dtype) for a in (wl.x, wl.residual, wl.weight))
    for variant in P.VARIANTS:
        sc = _scales_out(mode, n, 1024)
        q, sc, ro = rq.fused_add_rmsnorm_quant(x, r, w, wl.eps, mode, out_scales=sc, variant=variant)
        torch.cuda.synchronize()
        assert rq.take_fault_flags() == 0
        assert np.array_equal(q.cpu().numpy(), want["q"]), f"{mode}/{variant}: codes differ"
        assert np.array_equal(P.host_bits(ro), want["residual_out"])
        _check_scales(sc, want["scales"], mode, n, f"{mode}/{variant}")


@pytest.mark.parametrize("mode", OPTION_MODES)
def test_silu_mul_with_options(mode):
    act = ri.make_act_workload("opt_act", 37, 2048, seed=9)
    want = oracle.run_silu_mul(act.gate_up, mode=mode)
    gu = P.dev_act(act.gate_up, act.dtype)
    sc = _scales_out(mode, 37, 2048)
    q, sc = rq.silu_mul_quant(gu, mode, out_scales=sc)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want["q"])
    _check_scales(sc, want["scales"], mode, 37, mode)
