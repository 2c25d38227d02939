"""NVFP4 with a data-derived global scale (gs = 2688 / amax of y over the
batch) on the GPU, against the oracle's two-pass statement of it."""
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


def run_dyn(wl, variant, in_place=False, workspace=None):
    x = P.dev_act(wl.x, wl.dtype)
    r = None if wl.residual is None else P.dev_act(wl.residual, wl.dtype)
    w = P.dev_act(wl.weight, wl.dtype)
    q, sc, gs, ro = rq.fused_add_rmsnorm_nvfp4_dynamic(
        x, r, w, wl.eps, residual_out=r if (in_place and r is not None) else None,
        workspace=workspace, variant=variant)
    torch.cuda.synchronize()
    assert rq.take_fault_flags() == 0
    return {"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "global_scale": gs.cpu().numpy(),
            "residual_out": None if ro is None else P.host_bits(ro)}


def check_dyn(wl, label, **kw):
    want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=wl.dtype,
                                    nthreads=8)
    for v in P.VARIANTS:
        got = run_dyn(wl, v, **kw)
        assert got["global_scale"].view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0], \
            (label, v, got["global_scale"], want["global_scale"])
        P.compare(got, want, "nvfp4", f"{label}/{v}")


@pytest.mark.parametrize("n", ri.QWEN_TOKENS)
def test_qwen_shapes(n):
    check_dyn(ri.qwen_nvfp4(n), f"qwen_{n}")


@pytest.mark.parametrize("n", [1, 7, 64, 256])
def test_decode_fp16(n):
    check_dyn(ri.decode(n), f"decode_{n}")
    check_dyn(ri.decode(n, residual=False), f"decode_{n}_nores")


@pytest.mark.parametrize("H", [16, 48, 2064, 8192, 16384])
def test_ragged_hidden(H):
    for n in (1, 5, 700):
        check_dyn(ri.make_workload(f"dyn_{n}x{H}", n, H, res_sigma=1.5, seed=n + H), f"dyn_{n}x{H}")


def test_all_zero_batch_uses_unit_global_scale():
    wl = ri.Workload("zeros", 9, 256, "bf16", 1e-6, np.zeros((9, 256), np.uint16), None,
                     ri.to_bits(np.ones(256), "bf16"))
    for v in P.VARIANTS:
        got = run_dyn(wl, v)
        assert got["global_scale"][0] == 1.0 and not got["q"].any() and not got["scales"].any()


def test_in_place_and_reused_workspace():
    """The workspace is scratch: stale contents from another call must not leak."""
    ws = torch.full((rq.nvfp4_dynamic_workspace_bytes(4096),), 0x7F, dtype=torch.uint8, device="cuda")
    for seed in (1, 2):
        wl = ri.make_workload(f"inplace_{seed}", 300, 2048, res_sigma=1.0 + seed, seed=40 + seed)
        check_dyn(wl, f"inplace_{seed}", in_place=True, workspace=ws)


def test_workspace_too_small_is_rejected():
    x = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(rq.nvfp4_dynamic_workspace_bytes(8) - 16, dtype=torch.uint8, device="cuda")
    with pytest.raises(rq.RmsqError) as ei:
        rq.fused_add_rmsnorm_nvfp4_dynamic(x, None, w, 1e-6, workspace=ws)
    assert ei.value.status == rq.ERR_INVALID_ARG
