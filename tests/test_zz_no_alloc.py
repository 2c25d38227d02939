"""The allocation-free entry point of NVFP4 with a data-derived global scale.

It serves callers that cannot allocate device memory themselves; the library
keeps the workspace in a fixed device array instead.  Checked, through the C
ABI, against the entry point that takes a caller workspace, bit for bit (the
tolerance of every parity test here), on two calls in a row with different
inputs and shapes: the shared array keeps the first call's contents, so the
second call also shows that nothing stale leaks into its results.
"""
import ctypes

import numpy as np
import pytest
import torch

import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu

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


def test_noalloc_matches_workspace_entry_on_two_calls_in_a_row(rmsq_gpu):
    f = _entry()
    stream = torch.cuda.current_stream()
    cases = [ri.make_workload("noalloc_a", 700, 2048, res_sigma=2.0, seed=51),
             ri.make_workload("noalloc_b", 96, 4096, dtype="fp16", residual=False, seed=52)]
    for wl in cases:
        x, w = _dev(wl.x, wl.dtype), _dev(wl.weight, wl.dtype)
        r = None if wl.residual is None else _dev(wl.residual, wl.dtype)
        q_ref, sc_ref, gs_ref, ro_ref = rq.fused_add_rmsnorm_nvfp4_dynamic(x, r, w, wl.eps)

        n, H = wl.n_tokens, wl.hidden
        q = torch.empty_like(q_ref)
        sc = torch.empty_like(sc_ref)
        gs = torch.empty(1, dtype=torch.float32, device="cuda")
        ro = None if r is None else torch.empty_like(r)
        st = f(_p(x), _p(r), _p(w), ctypes.c_float(wl.eps), _p(q), _p(sc), _p(gs), _p(ro), n, H,
               0 if wl.dtype == "bf16" else 1, ctypes.c_void_p(stream.cuda_stream), 0)
        assert st == rq.OK, rq.status_string(st)
        torch.cuda.synchronize()
        assert torch.equal(q, q_ref), wl.name
        assert torch.equal(sc, sc_ref), wl.name
        assert gs.view(torch.int32).item() == gs_ref.view(torch.int32).item(), wl.name
        if ro is not None:
            assert torch.equal(ro.view(torch.int16), ro_ref.view(torch.int16)), wl.name


def test_noalloc_rejects_batches_beyond_its_array(rmsq_gpu):
    f = _entry()
    vp = ctypes.c_void_p
    fake = [vp(0x10000000 * k) for k in range(1, 8)]
    st = f(fake[0], None, fake[1], ctypes.c_float(1e-6), fake[2], fake[3], fake[4], None,
           MAX_TOKENS + 1, 64, 0, None, 0)
    assert st == rq.ERR_UNSUPPORTED_SHAPE
