"""The allocation-free entry point of NVFP4 with a data-derived global scale.

It serves callers that cannot allocate device memory themselves (a plugin
whose host engine owns every byte of device memory, code that must not call
cudaMalloc on a latency-critical path); the library keeps the workspace in a
fixed device array instead.  Checked through the C ABI against the oracle
(vLLM PR #51925 summary, "Motivation": block scales and FP4 values from the
normalised activations under an fp32 global scale, here taken from the data)
and against the entry point that takes a caller workspace, bit for bit (the
tolerance of every parity test here), on two calls in a row with different
inputs and shapes: the shared array keeps the first call's contents, so the
second call also shows that nothing stale leaks into its results.  A batch of
exactly the array's capacity is checked the same way.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

MAX_TOKENS = 65536      # RMSQ_NOALLOC_MAX_TOKENS in include/rmsq.h


def _entry():
    f = rq.load().rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc
    vp = ctypes.c_void_p
    f.argtypes = [vp, vp, vp, ctypes.c_float, vp, vp, vp, vp, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int, vp, ctypes.c_int]
    f.restype = ctypes.c_int
    return f


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(bits, dtype):
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(tdt).cuda()


def _bits(t):
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def _check_against_oracle_and_workspace_entry(f, wl):
    stream = torch.cuda.current_stream()
    x, w = _dev(wl.x, wl.dtype), _dev(wl.weight, wl.dtype)
    r = None if wl.residual is None else _dev(wl.residual, wl.dtype)
    n, H = wl.n_tokens, wl.hidden
    q = torch.empty(n, H // 2, dtype=torch.uint8, device="cuda")
    sc = torch.empty(n, H // 16, dtype=torch.uint8, device="cuda")
    gs = torch.empty(1, dtype=torch.float32, device="cuda")
    ro = None if r is None else torch.empty_like(r)
    st = f(_p(x), _p(r), _p(w), ctypes.c_float(wl.eps), _p(q), _p(sc), _p(gs), _p(ro), n, H,
           0 if wl.dtype == "bf16" else 1, ctypes.c_void_p(stream.cuda_stream), 0)
    assert st == rq.OK, rq.status_string(st)
    torch.cuda.synchronize()

    want = oracle.run_nvfp4_dynamic(wl.x, wl.residual, wl.weight, eps=wl.eps, dtype=wl.dtype, nthreads=16)
    assert gs.cpu().numpy().view(np.uint32)[0] == want["global_scale"].view(np.uint32)[0], wl.name
    assert np.array_equal(q.cpu().numpy(), want["q"]), wl.name
    assert np.array_equal(sc.cpu().numpy(), want["scales"]), wl.name
    if ro is not None:
        assert np.array_equal(_bits(ro), want["residual_out"]), wl.name

    q_ref, sc_ref, gs_ref, ro_ref = rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wl.eps)
    torch.cuda.synchronize()
    assert torch.equal(q, q_ref) and torch.equal(sc, sc_ref), wl.name
    assert gs.view(torch.int32).item() == gs_ref.view(torch.int32).item(), wl.name
    if ro is not None:
        assert torch.equal(ro.view(torch.int16), ro_ref.view(torch.int16)), wl.name


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_two_calls_in_a_row(rmsq_gpu):
    f = _entry()
    for wl in (ri.make_workload("noalloc_a", 700, 2048, res_sigma=2.0, seed=51),
               ri.make_workload("noalloc_b", 96, 4096, dtype="fp16", residual=False, seed=52)):
        _check_against_oracle_and_workspace_entry(f, wl)


@pytest.mark.gpu
def test_noalloc_at_its_largest_batch(rmsq_gpu):
    """Exactly RMSQ_NOALLOC_MAX_TOKENS rows: the per-row part of the array is
    used to its last entry."""
    f = _entry()
    _check_against_oracle_and_workspace_entry(
        f, ri.make_workload("noalloc_max", MAX_TOKENS, 64, res_sigma=1.5, seed=53))


def test_noalloc_rejects_batches_beyond_its_array():
    """Checked before any device access (runs without a GPU)."""
    f = _entry()
    vp = ctypes.c_void_p
    fake = [vp(0x10000000 * k) for k in range(1, 8)]
    st = f(fake[0], None, fake[1], ctypes.c_float(1e-6), fake[2], fake[3], fake[4], None,
           MAX_TOKENS + 1, 64, 0, None, 0)
    assert st == rq.ERR_UNSUPPORTED_SHAPE
    st = f(fake[0], None, fake[1], ctypes.c_float(1e-6), fake[2], fake[3], fake[4], None,
           MAX_TOKENS, 64, 7, None, 0)
    assert st == rq.ERR_INVALID_ARG        # a bad dtype is reported as for the workspace entry
