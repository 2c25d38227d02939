"""GPU parity on narrow rows with many row groups per CTA.

A row of 16 .. 512 elements (or 1024 with four chunks per thread) gives the
pipelined kernel one-warp CTAs, and a batch several times larger than its
persistent grid makes every CTA walk many row groups, so that both halves of
its double-buffered warp-sum slots are used.  Every quantisation mode (vLLM
docs "Fusion torch.compile passes", section "RMSNorm + Quantization
(fuse_norm_quant)", which puts no floor on the hidden size) and the
data-derived NVFP4 global scale, against the oracle, bf16 and fp16, with a row
count that is not a multiple of the grid.
"""
import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu

# 32 CTAs per SM x 152 SMs = 4864 one-warp CTAs at most: 16001 rows give each
# CTA three or four row groups, the last one ragged.
N_ROWS = 16001
GROUPS = {"fp8_group128_row": 128, "fp8_group128_col": 128, "fp8_group64_row": 64, "fp8_group64_col": 64}


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def _modes(H):
    return [m for m in rq.MODES if H % GROUPS.get(m, 16 if m == "nvfp4" else 8) == 0]


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("H,J", [(16, 0), (64, 0), (256, 0), (512, 0), (1024, 4)])
def test_one_warp_ctas_many_row_groups(H, J, dtype):
    wl = ri.make_workload(f"tiny_{H}", N_ROWS, H, dtype=dtype, res_sigma=1.7, seed=500 + H)
    rq.set_pipeline_config(J, 0, 0, 0)
    try:
        for mode in _modes(H):
            P.check(wl, mode, scale_in=0.06 if mode == "fp8_static" else None, nthreads=16,
                    variants=("pipelined", "auto"), label=f"tiny {N_ROWS}x{H} J{J} {dtype} {mode}")
        want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=dtype, nthreads=16)
        x, r, w = P.dev_act(wl.x, dtype), P.dev_act(wl.residual, dtype), P.dev_act(wl.weight, dtype)
        for variant in ("pipelined", "auto"):
            q, sc, gs, ro = rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wl.eps, variant=variant)
            torch.cuda.synchronize()
            assert rq.take_fault_flags() == 0
            assert gs.cpu().numpy().view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0]
            P.compare({"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "residual_out": P.host_bits(ro)},
                      want, "nvfp4", f"tiny dynamic {H} {dtype} {variant}")
    finally:
        rq.set_pipeline_config(0, 0, 0, 0)


@pytest.mark.parametrize("H", [16, 512])
def test_one_warp_ctas_without_residual(H):
    wl = ri.make_workload(f"tiny_nores_{H}", N_ROWS, H, residual=False, seed=600 + H)
    for mode in ("fp8_per_token", "nvfp4", "fp8_static"):
        P.check(wl, mode, scale_in=0.06 if mode == "fp8_static" else None, nthreads=16,
                variants=("pipelined",), label=f"tiny nores {H} {mode}")
