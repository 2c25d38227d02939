"""GPU parity of the all-reduce + residual add + RMSNorm + quantisation
kernel (vLLM docs "Fusion torch.compile passes", section "AllReduce + RMSNorm
(fuse_allreduce_rms)") against the oracle, bit for bit.

The ranks are emulated as separate buffers of this one device: the kernel's
loads from each rank's buffer are the same instructions that read peer
memory on a multi-GPU node, so the kernel code path under test is the one a
real run takes; only the addresses differ.
"""
import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu
MODES = list(rq.MODES) + ["fp8_group128_row+ue8m0", "fp8_per_token+e8m0"]


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def _partials(R, n, H, dtype, seed):
    return np.stack([ri.to_bits(ri.normal(seed + r, 1, n * H) * (0.5 + r % 3), dtype).reshape(n, H)
                     for r in range(R)])


def _scale(mode):
    return 0.05 if mode == "fp8_static" else None


def _run(parts, wl, mode, scale_in, in_place=False):
    dt = wl.dtype
    dev_parts = [P.dev_act(p, dt) for p in parts]
    r = None if wl.residual is None else P.dev_act(wl.residual, dt)
    w = P.dev_act(wl.weight, dt)
    s = torch.tensor([scale_in or 0.0], dtype=torch.float32, device="cuda")
    q, sc, ro = rq.allreduce_add_rmsnorm_quant(dev_parts, r, w, wl.eps, mode, s,
                                               residual_out=r if in_place else None)
    torch.cuda.synchronize()
    return {"q": q.cpu().numpy(), "scales": None if sc is None else sc.cpu().numpy(),
            "residual_out": None if ro is None else P.host_bits(ro)}


def _check(R, n, H, mode, dtype="bf16", residual=True, in_place=False, seed=0):
    wl = ri.make_workload(f"ar_{R}x{n}x{H}", n, H, dtype=dtype, residual=residual, res_sigma=1.5, seed=seed)
    parts = _partials(R, n, H, dtype, 100 + seed)
    scale_in = _scale(mode)
    if oracle.base_mode(mode) == "nvfp4":
        pre = oracle.run_allreduce(parts, wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token", dtype=dtype,
                                   want_y=True, nthreads=8)
        scale_in = oracle.nvfp4_global_scale(float(np.max(np.abs(pre["y"]))))
    want = oracle.run_allreduce(parts, wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=scale_in or 0.0,
                                dtype=dtype, nthreads=8)
    got = _run(parts, wl, mode, scale_in, in_place)
    if got["scales"] is not None and got["scales"].dtype == np.uint8 and want["scales"].dtype == np.uint8:
        assert np.array_equal(got["scales"], want["scales"]), mode
        got = dict(got, scales=None)
        want = dict(want, scales=None)
    return P.compare(got, want, oracle.base_mode(mode), f"allreduce R{R} n{n} H{H} {dtype} {mode}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("R", [1, 2, 8])
def test_modes_and_rank_counts(mode, R):
    for n, H in ((1, 4096), (7, 2048), (300, 8192)):
        _check(R, n, H, mode, seed=R * 10 + n)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("R", [3, 4])
def test_dtypes_without_residual_and_ragged_hidden(dtype, R):
    for H in (16, 1000, 4104, 16384):
        _check(R, 5, H, "fp8_per_token", dtype=dtype, residual=False, seed=H)
        _check(R, 5, H, "fp8_static", dtype=dtype, seed=H + 1)


def _pipelined_rows():
    """A batch that takes the pipelined kernel (from 4 rows per SM), with a ragged tail."""
    return 4 * torch.cuda.get_device_properties(0).multi_processor_count + 37


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("R", [1, 2, 4, 8])
def test_pipelined_kernel_modes_and_rank_counts(mode, R):
    """From 4 rows per SM and up to 4 ranks the pipelined kernel: every
    rank's partial row and the residual row copied into a shared-memory ring
    stage, summed there in rank order (8 ranks: the direct kernel)."""
    _check(R, _pipelined_rows(), 2048, mode, seed=R * 7 + 1)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("R", [3, 5])
def test_pipelined_kernel_dtypes_without_residual_and_ragged_hidden(dtype, R):
    n = _pipelined_rows()
    for H in (16, 1000, 4104):
        _check(R, n, H, "fp8_per_token", dtype=dtype, residual=False, seed=H)
        _check(R, n, H, "fp8_static", dtype=dtype, seed=H + 1)
    _check(R, n, 4096, "fp8_group64_row", dtype=dtype, residual=False, seed=2)


@pytest.mark.parametrize("shape", [(0, 0, 0), (4, 1, 0), (2, 1, 1), (0, 2, 2)],
                         ids=["default", "four-chunks-one-stage", "one-stage-one-cta-per-sm", "two-ctas-per-sm"])
def test_pipelined_kernel_many_rows_per_cta(shape):
    """Several rows per CTA (a wrapping ring), in place, under forced plans."""
    J, stages, cps = shape
    rq.set_pipeline_config(J, stages, cps, 0)
    try:
        _check(2, 3001, 2048, "fp8_static", in_place=True, seed=5)
        _check(4, 1500, 4096, "nvfp4", seed=6)
    finally:
        rq.set_pipeline_config(0, 0, 0, 0)


def test_rows_too_wide_for_the_ring_take_the_direct_kernel():
    """Four ranks' rows of hidden 16384 plus the residual exceed the ring
    budget: the direct kernel serves the batch, with the same results."""
    _check(4, _pipelined_rows(), 16384, "fp8_group128_row", seed=9)


def test_in_place_residual_update():
    _check(2, 64, 4096, "nvfp4", in_place=True, seed=5)
    _check(4, 64, 4096, "fp8_group64_col", in_place=True, seed=6)


def test_two_shot_row_slices_equal_the_one_shot_result():
    """Each emulated rank reduces and normalises its own slice of the rows
    (the pointers and row count of the slice), then the slices are put back
    together: identical to every row done at once."""
    R, n, H, mode = 4, 103, 2048, "fp8_per_token"
    wl = ri.make_workload("ar_two_shot", n, H, res_sigma=1.5, seed=9)
    parts = _partials(R, n, H, "bf16", 200)
    whole = _run(parts, wl, mode, None)
    dev_parts = [P.dev_act(p, "bf16") for p in parts]
    r = P.dev_act(wl.residual, "bf16")
    w = P.dev_act(wl.weight, "bf16")
    q = torch.empty(n, H, dtype=torch.uint8, device="cuda")
    sc = torch.empty(n, dtype=torch.float32, device="cuda")
    ro = torch.empty_like(r)
    for rank in range(R):
        b, e = rq.row_slice(n, R, rank)
        rq.allreduce_add_rmsnorm_quant([p[b:e] for p in dev_parts], r[b:e], w, wl.eps, mode,
                                       out_q=q[b:e], out_scales=sc[b:e], residual_out=ro[b:e])
    torch.cuda.synchronize()
    assert np.array_equal(q.cpu().numpy(), whole["q"])
    assert np.array_equal(sc.cpu().numpy().view(np.uint32), whole["scales"].view(np.uint32))
    assert np.array_equal(P.host_bits(ro), whole["residual_out"])


def test_argument_errors():
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ValueError):
        rq.allreduce_add_rmsnorm_quant([], None, w, 1e-6, "fp8_per_token")
    with pytest.raises(ValueError):
        rq.allreduce_add_rmsnorm_quant([x] * 9, None, w, 1e-6, "fp8_per_token")
    buf = torch.zeros(4 * 64 * 2, dtype=torch.uint8, device="cuda")
    part = buf.view(torch.bfloat16).view(4, 64)
    with pytest.raises(rq.RmsqError) as ei:     # the codes would overwrite a rank's partials
        rq.allreduce_add_rmsnorm_quant([x, part], None, w, 1e-6, "fp8_per_token", out_q=buf[:256].view(4, 64))
    assert ei.value.status == rq.ERR_ALIAS
