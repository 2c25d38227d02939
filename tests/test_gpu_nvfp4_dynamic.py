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


@pytest.mark.parametrize("n,H", [(3001, 2064), (50001, 48), (2500, 7168)])
def test_second_pass_column_walk(n, H):
    """The second pass gives each thread one column of 16-element blocks and
    walks it down the rows at a stride of R rows: an odd number of blocks
    per row (129, 3, 448) and several rows per thread, with the last pair
    of rows ragged."""
    check_dyn(ri.make_workload(f"walk_{n}x{H}", n, H, res_sigma=1.0, seed=n + H), f"walk_{n}x{H}")


def test_second_pass_column_walk_fp16_without_residual():
    """The same walk over x itself (no residual) in fp16."""
    wl = ri.make_workload("walk_fp16_nores", 5000, 2048, dtype="fp16", residual=False, seed=77)
    check_dyn(wl, "walk_fp16_nores")


def test_all_zero_batch_uses_unit_global_scale():
    wl = ri.Workload("zeros", 9, 256, "bf16", 1e-6, np.zeros((9, 256), np.uint16), None,
                     ri.to_bits(np.ones(256), "bf16"))
    for v in P.VARIANTS:
        got = run_dyn(wl, v)
        assert got["global_scale"][0] == 1.0 and not got["q"].any() and not got["scales"].any()


@pytest.mark.parametrize("fill", [0x00, 0x7F, 0xFF])
def test_in_place_and_reused_workspace(fill):
    """The workspace is scratch: neither its contents on entry (a constant
    byte) nor what another call left there may leak into a call."""
    ws = torch.full((rq.nvfp4_dynamic_workspace_bytes(4096),), fill, dtype=torch.uint8, device="cuda")
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


@pytest.mark.parametrize("shape", [(1, 0), (2, 1), (0, 1)], ids=["one-cta-per-sm", "two-ctas-one-stage",
                                                                 "one-stage"])
def test_pipelined_first_pass_with_small_grids(shape):
    """Pass 1 on the pipelined kernel with fewer resident CTAs or ring stages
    than usual (many rows per CTA)."""
    cps, stages = shape
    wl = ri.qwen_nvfp4(4096)
    want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=wl.dtype, nthreads=8)
    rq.set_pipeline_config(0, stages, cps, 0)
    try:
        got = run_dyn(wl, "pipelined")
    finally:
        rq.set_pipeline_config(0, 0, 0, 0)
    assert got["global_scale"].view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0]
    P.compare(got, want, "nvfp4", f"small grid {shape}")


@pytest.mark.parametrize("variant", ["auto", "direct"])
def test_graph_replay_resets_the_workspace(variant):
    """Captured once into a CUDA graph and replayed on new inputs: each replay
    writes every workspace entry it reads (inverse RMS, per-CTA maxima)."""
    wls = [ri.make_workload(f"graph{i}", 900, 2048, res_sigma=1.0 + i, seed=300 + i) for i in range(3)]
    x = P.dev_act(wls[0].x, wls[0].dtype)
    r = P.dev_act(wls[0].residual, wls[0].dtype)
    w = P.dev_act(wls[0].weight, wls[0].dtype)
    n, H = x.shape
    q = torch.empty(n, H // 2, dtype=torch.uint8, device="cuda")
    sc = torch.empty(n, H // 16, dtype=torch.uint8, device="cuda")
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    ro = torch.empty_like(r)
    ws = torch.empty(rq.nvfp4_dynamic_workspace_bytes(n), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()

    def call():
        rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wls[0].eps, out_q=q, out_scales=sc, out_global_scale=gs,
                                           residual_out=ro, workspace=ws, stream=s, variant=variant)

    with torch.cuda.stream(s):
        call()   # first call outside capture (library set-up)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call()
    for wl in wls:
        x.copy_(P.dev_act(wl.x, wl.dtype))
        r.copy_(P.dev_act(wl.residual, wl.dtype))
        w.copy_(P.dev_act(wl.weight, wl.dtype))
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert rq.take_fault_flags() == 0
        want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=wl.dtype, nthreads=8)
        got = {"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "global_scale": gs.cpu().numpy(),
               "residual_out": P.host_bits(ro)}
        assert got["global_scale"].view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0]
        P.compare(got, want, "nvfp4", f"graph replay {wl.name}/{variant}")


@pytest.mark.parametrize("pdl", [True, False], ids=["pdl", "plain"])
@pytest.mark.parametrize("variant", ["auto", "direct"])
def test_back_to_back_calls_share_a_workspace(variant, pdl):
    """Three calls queued on one stream with one workspace and no host
    synchronisation between them, with and without programmatic dependent
    launch: each call's first pass must not overwrite the per-CTA maxima
    before the previous call's second pass has read them."""
    wls = [ri.make_workload(f"b2b{i}", 4096, 2048, res_sigma=0.5 + i, seed=500 + i) for i in range(3)]
    ws = torch.full((rq.nvfp4_dynamic_workspace_bytes(4096),), 0x7F, dtype=torch.uint8, device="cuda")
    ins = [(P.dev_act(wl.x, wl.dtype), P.dev_act(wl.residual, wl.dtype), P.dev_act(wl.weight, wl.dtype))
           for wl in wls]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    outs = []
    rq.set_programmatic_launch(pdl)
    try:
        for wl, (x, r, w) in zip(wls, ins):
            outs.append(rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wl.eps, workspace=ws, stream=s,
                                                           variant=variant))
        torch.cuda.synchronize()
    finally:
        rq.set_programmatic_launch(True)
    assert rq.take_fault_flags() == 0
    for wl, (q, sc, gs, ro) in zip(wls, outs):
        want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=wl.dtype, nthreads=8)
        got = {"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "global_scale": gs.cpu().numpy(),
               "residual_out": P.host_bits(ro)}
        assert got["global_scale"].view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0], wl.name
        P.compare(got, want, "nvfp4", f"back to back {wl.name}/{variant}")
