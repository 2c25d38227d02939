"""The two ops of the unfused sequence on the GPU against the oracle, bit for
bit: the norm alone (y in the activation type, residual write-back) and the
quantisation of an activation-type tensor in every mode and scale option."""
import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("n,H,residual", [(7, 4096, True), (1500, 4096, True), (1500, 2048, False),
                                          (3, 12288, True), (900, 7168, True)])
def test_norm_alone(dtype, n, H, residual):
    wl = ri.make_workload(f"na_{n}x{H}", n, H, dtype=dtype, residual=residual, res_sigma=1.5, seed=n + H)
    want = oracle.run_add_rmsnorm(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=dtype, nthreads=8)
    x = P.dev_act(wl.x, dtype)
    r = None if wl.residual is None else P.dev_act(wl.residual, dtype)
    w = P.dev_act(wl.weight, dtype)
    y, ro = rq.fused_add_rmsnorm(x, r, w, wl.eps)
    torch.cuda.synchronize()
    assert rq.take_fault_flags() == 0
    assert np.array_equal(P.host_bits(y), want["y_t"])
    if residual:
        assert np.array_equal(P.host_bits(ro), want["residual_out"])


@pytest.mark.parametrize("mode", ["fp8_static", "fp8_per_token", "fp8_group128_row", "fp8_group128_col",
                                  "fp8_group64_row", "fp8_group64_col", "nvfp4", "fp8_group128_col+e8m0+tma"])
def test_quant_alone(mode):
    wl = ri.make_workload("qa", 300, 4096, res_sigma=2.0, seed=12)
    y_t = oracle.run_add_rmsnorm(wl.x, wl.residual, wl.weight, eps=wl.eps, nthreads=8)["y_t"]
    scale_in = {"fp8_static": 0.05, "nvfp4": 2688.0 / 9.0}.get(mode, 0.0)
    want = oracle.run_quant(y_t, mode=mode, scale_in=scale_in, nthreads=8)
    s = torch.tensor([scale_in], dtype=torch.float32, device="cuda")
    q, sc = rq.quant(P.dev_act(y_t, "bf16"), mode, s)
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), want["q"])
    if sc is not None:
        g = sc.cpu().numpy()
        w = want["scales"]
        if "+tma" in mode:
            g, w = g[:, :300], w[:, :300]
        assert np.array_equal(g.view(np.uint8), w.view(np.uint8))


def test_unfused_sequence_on_the_llama_layer():
    """Both ops back to back on the Llama-8B-shaped layer (4096 x 4096, per-token)."""
    wl = ri.llama(4096, True)
    y = oracle.run_add_rmsnorm(wl.x, wl.residual, wl.weight, eps=wl.eps, nthreads=16)
    want = oracle.run_quant(y["y_t"], mode="fp8_per_token", nthreads=16)
    x, r, w = (P.dev_act(a, wl.dtype) for a in (wl.x, wl.residual, wl.weight))
    yd, ro = rq.fused_add_rmsnorm(x, r, w, wl.eps)
    q, sc = rq.quant(yd, "fp8_per_token")
    torch.cuda.synchronize()
    assert np.array_equal(P.host_bits(ro), y["residual_out"])
    assert np.array_equal(q.cpu().numpy(), want["q"])
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), want["scales"].view(np.uint32))
