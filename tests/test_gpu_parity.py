"""GPU parity: the CUDA path through the C ABI against the CPU oracle, element by
element, on the same seeded inputs.

Covers the five workloads of the path (the 64x512 static-FP8 case, the
Llama-, DeepSeek-V3- and Qwen3-shaped layers, the fp16 decode sweep) at the
sizes the benchmark launches, plus ragged / tiny / maximum shapes, in-place
residual updates, and the hand-worked rows.
"""
import json
import os

import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu

ALL_MODES = list(rq.MODES)
GROUP_MODES = ["fp8_group128_row", "fp8_group128_col", "fp8_group64_row", "fp8_group64_col"]
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "worked_examples.json")


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


# ---------------------------------------------------------------- worked rows
def _golden():
    return [e for e in json.load(open(GOLDEN))["examples"] if e["H"] % 8 == 0]


@pytest.mark.parametrize("ex", _golden(), ids=lambda e: e["name"])
def test_golden_rows_on_gpu(ex):
    n, H = ex["n"], ex["H"]

    def fill(v, shape):
        a = np.asarray(v, np.float64)
        return np.broadcast_to(a, shape).copy() if a.size == 1 else a.reshape(shape)

    x = ri.to_bits(fill(ex["x"], (n, H)), ex["dtype"]).reshape(n, H)
    r = None if ex["residual"] is None else ri.to_bits(fill(ex["residual"], (n, H)), ex["dtype"]).reshape(n, H)
    w = ri.to_bits(fill(ex["weight"], (H,)), ex["dtype"])
    wl = ri.Workload(ex["name"], n, H, ex["dtype"], ex["eps"], x, r, w)
    for variant in P.VARIANTS:
        got = P.run_gpu(wl, ex["mode"], ex["scale_in"], variant=variant)
        q = got["q"].ravel()
        b = bytes.fromhex(ex["expect"]["q_hex"])
        want = np.frombuffer(b * (q.size // len(b)) if len(b) < q.size else b, np.uint8)
        assert np.array_equal(q, want), (variant, q.tobytes().hex(), ex["expect"]["q_hex"])
        e = ex["expect"]
        if "residual_out_hex" in e:
            assert np.all(got["residual_out"] == int(e["residual_out_hex"], 16))
        if "scales_f32_bits" in e:
            assert np.all(got["scales"].view(np.uint32) == int(e["scales_f32_bits"][0], 16))
        if "scales_u8_hex" in e:
            assert np.all(got["scales"] == int(e["scales_u8_hex"][0], 16))


# ---------------------------------------------------------------- the five workloads
def test_pr1_static_fp8():
    P.check(ri.pr1(), "fp8_static")


@pytest.mark.parametrize("residual", [True, False], ids=["res", "nores"])
def test_llama_per_token_full_size(residual):
    P.check(ri.llama(4096, residual=residual), "fp8_per_token", nthreads=16)


@pytest.mark.parametrize("mode", ALL_MODES)
def test_llama_shape_every_mode(mode):
    P.check(ri.llama(512), mode, scale_in=0.1 if mode == "fp8_static" else None)


@pytest.mark.parametrize("mode", GROUP_MODES)
def test_dsv3_groups_full_size(mode):
    P.check(_dsv3_full(), mode, nthreads=16)


_DSV3 = {}


def _dsv3_full():
    if "wl" not in _DSV3:
        _DSV3["wl"] = ri.dsv3(8192)
    return _DSV3["wl"]


@pytest.mark.parametrize("n", ri.QWEN_TOKENS)
def test_qwen_nvfp4(n):
    P.check(ri.qwen_nvfp4(n), "nvfp4", nthreads=16)


@pytest.mark.parametrize("residual", [True, False], ids=["res", "nores"])
@pytest.mark.parametrize("mode", ["fp8_static", "fp8_per_token", "fp8_group128_row", "nvfp4"])
def test_decode_sweep(mode, residual):
    for n in ri.DECODE_TOKENS:
        P.check(ri.decode(n, residual=residual), mode, label=f"decode_{n}/{mode}/{residual}")


# ---------------------------------------------------------------- edges
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("H", [8, 16, 24, 136, 1000, 4104, 8200, 16384])
def test_ragged_and_maximum_hidden(dtype, H):
    for n in (1, 3, 33):
        wl = ri.make_workload(f"rag_{n}x{H}", n, H, dtype=dtype, res_sigma=1.5, seed=H + n)
        for mode in ALL_MODES:
            if mode == "nvfp4" and H % 16:
                continue
            if mode in GROUP_MODES and H % (128 if "128" in mode else 64):
                continue
            P.check(wl, mode, scale_in=0.07 if mode == "fp8_static" else None,
                    label=f"{wl.name}/{dtype}/{mode}")


def test_empty_input_launches_nothing():
    x = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    q, sc, ro = rq.fused_add_rmsnorm_quant(x, x, w, 1e-6, "fp8_per_token")
    assert q.numel() == 0 and sc.numel() == 0 and ro.numel() == 0


def test_in_place_residual_update():
    wl = ri.make_workload("inplace", 40, 2048, seed=31)
    for mode in ("fp8_per_token", "nvfp4", "fp8_group64_col"):
        P.check(wl, mode, in_place=True, label=f"inplace/{mode}")


def test_residual_out_over_x():
    wl = ri.make_workload("over_x", 9, 1024, seed=32)
    want = oracle.run_workload(wl, "fp8_per_token")
    x = P.dev_act(wl.x, "bf16")
    r = P.dev_act(wl.residual, "bf16")
    w = P.dev_act(wl.weight, "bf16")
    q, sc, ro = rq.fused_add_rmsnorm_quant(x, r, w, wl.eps, "fp8_per_token", residual_out=x)
    torch.cuda.synchronize()
    assert ro.data_ptr() == x.data_ptr()
    P.compare({"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "residual_out": P.host_bits(x)},
              want, "fp8_per_token", "residual_out=x")


def test_guard_bands_and_determinism():
    """Outputs inside larger sentinel-filled buffers: nothing outside the
    documented extents is written, and two runs give identical bytes."""
    n, H = 77, 2048
    wl = ri.make_workload("guard", n, H, seed=33)
    x = P.dev_act(wl.x, "bf16")
    r = P.dev_act(wl.residual, "bf16")
    w = P.dev_act(wl.weight, "bf16")
    G = 4096
    for mode in ALL_MODES:
        qb, sb = rq.query_sizes(mode, n, H)
        outs = []
        for rep in range(2):
            qbuf = torch.full((qb + 2 * G,), 0xA5, dtype=torch.uint8, device="cuda")
            sbuf = torch.full((sb + 2 * G,), 0x5A, dtype=torch.uint8, device="cuda")
            rbuf = torch.full((n * H + 2 * G,), -12345, dtype=torch.int16, device="cuda")
            q = qbuf[G:G + qb].view(n, -1)
            sc = None if sb == 0 else sbuf[G:G + sb]
            if sc is not None and mode != "nvfp4":
                sc = sc.view(torch.float32)
            ro = rbuf[G:G + n * H].view(torch.bfloat16).view(n, H)
            s_in = torch.tensor([0.05 if mode == "fp8_static" else 300.0], device="cuda")
            rq.fused_add_rmsnorm_quant(x, r, w, 1e-6, mode, s_in, out_q=q, out_scales=sc, residual_out=ro)
            torch.cuda.synchronize()
            for buf, fill in ((qbuf, 0xA5), (sbuf, 0x5A)):
                assert torch.all(buf[:G] == fill) and torch.all(buf[-G:] == fill), mode
            assert torch.all(rbuf[:G] == -12345) and torch.all(rbuf[-G:] == -12345), mode
            outs.append((qbuf.cpu(), sbuf.cpu(), rbuf.cpu()))
        for a, b in zip(outs[0], outs[1]):
            assert torch.equal(a, b), mode


def test_misaligned_pointers_rejected_before_launch():
    x = torch.zeros(4 * 64 + 8, dtype=torch.bfloat16, device="cuda")
    w = torch.ones(64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rq.RmsqError) as ei:
        rq.fused_add_rmsnorm_quant(x[4:4 + 256].view(4, 64), None, w, 1e-6, "fp8_per_token")
    assert ei.value.status == rq.ERR_ALIGNMENT


def test_non_default_stream():
    wl = ri.make_workload("stream", 50, 4096, seed=34)
    s = torch.cuda.Stream()
    want = oracle.run_workload(wl, "fp8_group128_row")
    with torch.cuda.stream(s):
        got = P.run_gpu(wl, "fp8_group128_row", None, stream=s)
    P.compare(got, want, "fp8_group128_row", "side stream")


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_subnormal_zero_and_wide_range_inputs(dtype):
    """Log-uniform magnitudes from the subnormal range of the activation type
    up to 2^10, random signs, exact +-0: the packed residual add, the squares
    and the quantisation must still match the oracle bit for bit."""
    n, H = 64, 1024
    u = ri.uniform(77, 1, 3 * n * H)
    lo = -133.0 if dtype == "bf16" else -24.0
    mag = 2.0 ** (lo + (10.0 - lo) * u[: 2 * n * H])
    sign = np.where(u[n * H: 3 * n * H] < 0.5, -1.0, 1.0)
    vals = mag * sign
    vals[::97] = 0.0
    vals[1::101] = -0.0
    x = ri.to_bits(vals[: n * H], dtype).reshape(n, H)
    r = ri.to_bits(vals[n * H:], dtype).reshape(n, H)
    w = ri.to_bits(1.0 + 0.1 * ri.normal(78, 1, H), dtype)
    wl = ri.Workload(f"wide_{dtype}", n, H, dtype, 1e-6, x, r, w)
    for mode in ("fp8_static", "fp8_per_token", "fp8_group64_row", "nvfp4"):
        P.check(wl, mode, scale_in=0.5 if mode == "fp8_static" else None, label=f"wide/{dtype}/{mode}")


def test_static_scale_sweep():
    """Many static scales (including subnormal-ratio and saturating ones):
    exercises the bracketing reciprocal and its exact fallback across scales."""
    wl = ri.make_workload("sweep", 16, 512, res_sigma=1.3, seed=37)
    u = ri.uniform(38, 1, 120)
    scales = np.float32(10.0) ** (-8.0 + 14.0 * u).astype(np.float32)
    for s in list(scales) + [np.float32(1.0), np.float32(0.1), np.float32(2.0 ** -20)]:
        P.check(wl, "fp8_static", scale_in=float(s), label=f"static s={float(s):.3e}")


@pytest.mark.parametrize("mode", ["fp8_group64_col", "fp8_per_token", "nvfp4", "fp8_static"])
def test_pipelined_launch_shapes_do_not_change_results(mode):
    """Chunks per thread (1 to 8: one to sixteen warps per row), ring depth and
    CTAs per SM, on an odd row count; the rows-per-iteration setting is
    accepted and changes nothing."""
    wl = ri.make_workload("shapes", 701, 4096, res_sigma=2.0, seed=36)
    s_in = 0.05 if mode == "fp8_static" else None
    want = oracle.run_workload(wl, mode, scale_in=s_in, nthreads=8)
    try:
        for J, stages, cps, rows in ((1, 2, 1, 1), (2, 1, 2, 1), (4, 8, 3, 1), (2, 6, 0, 0), (0, 3, 4, 1),
                                     (2, 2, 0, 2), (1, 1, 2, 2), (2, 3, 1, 2), (4, 2, 0, 2), (8, 2, 0, 0),
                                     (8, 1, 12, 0), (4, 3, 20, 0)):
            rq.set_pipeline_config(J, stages, cps, rows)
            got = P.run_gpu(wl, mode, want["scale_in"], variant="pipelined")
            P.compare(got, want, mode, f"{mode} shape J{J} s{stages} c{cps} r{rows}")
    finally:
        rq.set_pipeline_config(0, 0, 0, 0)


def test_nvfp4_dynamic_with_two_rows_per_iteration():
    wl = ri.make_workload("dyn_r2", 1233, 2048, res_sigma=1.5, seed=39)
    want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, nthreads=8)
    x, r, w = P.dev_act(wl.x, "bf16"), P.dev_act(wl.residual, "bf16"), P.dev_act(wl.weight, "bf16")
    try:
        for rows in (1, 2):
            rq.set_pipeline_config(0, 0, 0, rows)
            q, sc, gs, ro = rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wl.eps, variant="pipelined")
            torch.cuda.synchronize()
            assert gs.cpu().numpy().view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0]
            P.compare({"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "residual_out": P.host_bits(ro)},
                      want, "nvfp4", f"dynamic r{rows}")
    finally:
        rq.set_pipeline_config(0, 0, 0, 0)


def test_pipelined_ring_sizes_in_any_order():
    """One pipelined instantiation launched with shrinking and growing rings."""
    for H in (16, 8, 2048, 8, 16, 2048):
        wl = ri.make_workload(f"ring_{H}", 5, H, seed=35 + H)
        P.check(wl, "fp8_per_token", variants=("pipelined",), label=f"ring/{H}")


@pytest.mark.parametrize("mode", ["fp8_per_token", "fp8_group128_row", "nvfp4"])
@pytest.mark.parametrize("H", [4096, 12288])
def test_sixteen_byte_aligned_buffers(mode, H):
    """Buffers that start on 16 but not 32 bytes take the per-chunk loads and
    stores instead of the paired 32-byte accesses; results stay bit-exact."""
    n = 700
    wl = ri.make_workload("align16", n, H, seed=51)
    want = oracle.run_workload(wl, mode)
    scale_in = want["scale_in"]
    qcols = H // 2 if mode == "nvfp4" else H

    def shifted(numel, dtype):
        # 16 bytes past a 256-byte aligned allocation
        per = 16 // torch.empty((), dtype=dtype).element_size()
        return torch.zeros(numel + per, dtype=dtype, device="cuda")[per:]

    for variant in P.VARIANTS:
        x = shifted(n * H, torch.bfloat16).view(n, H)
        x.copy_(P.dev_act(wl.x, wl.dtype))
        r = shifted(n * H, torch.bfloat16).view(n, H)
        r.copy_(P.dev_act(wl.residual, wl.dtype))
        ro = shifted(n * H, torch.bfloat16).view(n, H)
        q = shifted(n * qcols, torch.uint8).view(n, qcols)
        assert x.data_ptr() % 32 == 16 and q.data_ptr() % 32 == 16
        w = P.dev_act(wl.weight, wl.dtype)
        s = torch.tensor([scale_in or 0.0], dtype=torch.float32, device="cuda")
        q, sc, ro = rq.fused_add_rmsnorm_quant(x, r, w, wl.eps, mode, s, out_q=q, residual_out=ro,
                                               variant=variant)
        torch.cuda.synchronize()
        assert rq.take_fault_flags() == 0
        got = {"q": q.cpu().numpy(), "scales": sc.cpu().numpy(), "residual_out": P.host_bits(ro)}
        P.compare(got, want, mode, f"16-byte aligned {variant}")


@pytest.mark.parametrize("n", [40, 1300], ids=["direct", "pipelined"])
@pytest.mark.parametrize("pdl", [True, False], ids=["pdl", "plain"])
def test_chained_layers_in_place(n, pdl):
    """Four back-to-back calls on one stream, as consecutive layers: each
    reads the residual the previous one wrote (odd layers update it in
    place), with no host synchronisation in between.  With programmatic dependent launch each
    kernel must still see the previous one's writes; the oracle applies the
    layers one after the other."""
    H, layers = 2048, 4
    wls = [ri.make_workload(f"chain{i}", n, H, res_sigma=2.0, seed=90 + i) for i in range(layers)]
    mode = "fp8_per_token"
    # oracle: residual carried from layer to layer
    res_bits = wls[0].residual
    want = []
    for wl in wls:
        out = oracle.run(wl.x, res_bits, wl.weight, eps=wl.eps, mode=mode, dtype=wl.dtype)
        want.append(out)
        res_bits = out["residual_out"]
    rq.set_programmatic_launch(pdl)
    try:
        s = torch.cuda.Stream()
        xs = [P.dev_act(wl.x, wl.dtype) for wl in wls]
        ws = [P.dev_act(wl.weight, wl.dtype) for wl in wls]
        # even layers write a fresh buffer, odd layers update it in place
        bufs = [P.dev_act(wls[0].residual, wls[0].dtype)] + [torch.empty_like(xs[0]) for _ in range(layers // 2)]
        torch.cuda.synchronize()
        outs = []
        r = bufs[0]
        with torch.cuda.stream(s):
            for i in range(layers):
                ro = bufs[i // 2 + 1]
                q, sc, _ = rq.fused_add_rmsnorm_quant(xs[i], r, ws[i], wls[i].eps, mode, residual_out=ro,
                                                      stream=s)
                outs.append((q, sc, ro if i % 2 == 1 else None))
                r = ro
        torch.cuda.synchronize()
    finally:
        rq.set_programmatic_launch(True)
    assert rq.take_fault_flags() == 0
    for i, (q, sc, ro) in enumerate(outs):
        # an even layer's write-back is overwritten in place by the next layer
        got = {"q": q.cpu().numpy(), "scales": sc.cpu().numpy(),
               "residual_out": None if ro is None else P.host_bits(ro)}
        w = dict(want[i])
        if ro is None:
            w["residual_out"] = None
        P.compare(got, w, mode, f"layer {i}")
