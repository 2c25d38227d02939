"""Scale options on the GPU (E8M0 power-of-two scales, their UE8M0 bytes,
TMA-aligned column-major stride) against the oracle (blog "[vLLM]
Compilation Fusion Passes", section "Why this design", item 3): bit for bit
for the norm op in every kernel variant, and for SiLU+Mul bit for bit against
the quantisation of the kernel's own activations (within the activation bar
against the independent oracle); padding entries of the aligned layout are
not written."""
import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri
from test_gpu_act import ACT_SCALE_ULP, kernel_activations

pytestmark = pytest.mark.gpu
OPTION_MODES = ["fp8_per_token+e8m0", "fp8_group128_row+e8m0", "fp8_group64_col+e8m0",
                "fp8_group128_col+tma", "fp8_group64_col+e8m0+tma",
                "fp8_per_token+ue8m0", "fp8_group128_row+ue8m0", "fp8_group64_row+ue8m0",
                "fp8_group128_col+ue8m0", "fp8_group64_col+ue8m0+tma"]
SENTINEL = 0x7f


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def _scales_out(mode, n, H):
    sc = rq.scales_like(mode, n, H, "cuda")
    sc.view(torch.uint8).fill_(SENTINEL)
    return sc


def _check_scales(got_sc, want_sc, mode, n, label):
    g = got_sc.cpu().numpy()
    assert g.dtype == want_sc.dtype and g.shape == want_sc.shape, (g.dtype, want_sc.dtype, g.shape, want_sc.shape)
    if "+tma" in mode:
        assert np.all(g[:, n:].view(np.uint8) == SENTINEL), f"{label}: padding written"
        g, want_sc = g[:, :n], want_sc[:, :n]
    assert np.array_equal(g.view(np.uint8), want_sc.view(np.uint8)), f"{label}: scales differ"


@pytest.mark.parametrize("mode", OPTION_MODES)
@pytest.mark.parametrize("n", [13, 900, 5000])
def test_norm_op_with_options(mode, n):
    wl = ri.make_workload(f"opt_{n}", n, 1024, res_sigma=1.5, seed=n)
    want = oracle.run_workload(wl, mode, nthreads=8)
    x, r, w = (P.dev_act(a, wl.dtype) for a in (wl.x, wl.residual, wl.weight))
    for variant in P.VARIANTS:
        sc = _scales_out(mode, n, 1024)
        q, sc, ro = rq.fused_add_rmsnorm_quant(x, r, w, wl.eps, mode, out_scales=sc, variant=variant)
        torch.cuda.synchronize()
        assert rq.take_fault_flags() == 0
        assert np.array_equal(q.cpu().numpy(), want["q"]), f"{mode}/{variant}: codes differ"
        assert np.array_equal(P.host_bits(ro), want["residual_out"])
        _check_scales(sc, want["scales"], mode, n, f"{mode}/{variant}")


@pytest.mark.parametrize("mode", ["fp8_per_token+ue8m0", "fp8_group128_col+ue8m0+tma"])
def test_quant_alone_with_byte_scales(mode):
    """The unfused quantisation entry point takes the same option."""
    wl = ri.make_workload("opt_q", 77, 2048, seed=12)
    y = oracle.run_add_rmsnorm(wl.x, wl.residual, wl.weight, eps=wl.eps)["y_t"]
    want = oracle.run_quant(y, mode=mode)
    sc = _scales_out(mode, 77, 2048)
    q, sc = rq.quant(P.dev_act(y, wl.dtype), mode, out_scales=sc)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want["q"])
    _check_scales(sc, want["scales"], mode, 77, mode)


@pytest.mark.parametrize("mode", OPTION_MODES)
def test_silu_mul_with_options(mode):
    act = ri.make_act_workload("opt_act", 37, 2048, seed=9)
    gu = P.dev_act(act.gate_up, act.dtype)
    sc = _scales_out(mode, 37, 2048)
    q, sc = rq.silu_mul_quant(gu, mode, out_scales=sc)
    torch.cuda.synchronize()
    # exact: the option applied to the kernel's own activations
    mine = oracle.run_quant_f32(kernel_activations(act), mode=mode)
    assert np.array_equal(q.cpu().numpy(), mine["q"])
    _check_scales(sc, mine["scales"], mode, 37, mode)
    # and within the activation bar of the independent oracle
    want = oracle.run_silu_mul(act.gate_up, mode=mode)
    steps = P.code_steps(q.cpu().numpy(), want["q"], "fp8_static")
    assert steps.max() <= 1 and np.count_nonzero(steps) <= P.MAX_MISMATCH_FRAC * steps.size + 1
    g, w = sc.cpu().numpy(), want["scales"]
    if "+tma" in mode:
        g, w = g[:, :37], w[:, :37]
    if g.dtype == np.uint8:     # a power-of-two scale moves by at most one binade
        assert np.max(np.abs(g.astype(np.int64) - w.astype(np.int64))) <= 1
    else:
        assert np.max(np.abs(g.view(np.int32).astype(np.int64) - w.view(np.int32).astype(np.int64))) <= ACT_SCALE_ULP
