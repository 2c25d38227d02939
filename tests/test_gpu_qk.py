"""QK-norm + RoPE on the GPU against the oracle, bit for bit (every q / k head,
v untouched, out-of-range positions left unchanged)."""
import dataclasses

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


VARIANTS = ["direct", "pipelined"]


def run_gpu(wl, variant="auto"):
    qkv = P.dev_act(wl.qkv, wl.dtype)
    pos = torch.from_numpy(wl.positions).cuda()
    cs = torch.from_numpy(wl.cos_sin).cuda()
    qw, kw = P.dev_act(wl.q_weight, wl.dtype), P.dev_act(wl.k_weight, wl.dtype)
    rq.qk_norm_rope(qkv, pos, cs, qw, kw, wl.eps, wl.nq, wl.nkv, wl.head_dim, wl.neox, variant=variant)
    torch.cuda.synchronize()
    return P.host_bits(qkv)


def check(wl, variant="auto", want=None):
    want = oracle.run_qk_norm_rope(wl) if want is None else want
    got = run_gpu(wl, variant)
    bad = np.count_nonzero(got != want)
    assert bad == 0, f"{wl.name} ({variant}): {bad} of {want.size} elements differ"
    assert rq.take_fault_flags() == 0


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_qwen_attention_shape(neox):
    """4096 tokens, 32 q heads, 4 kv heads, head_dim 128 (Qwen3-30B-A3B), in
    the launch the bench times (auto: pipelined) and the warp kernel."""
    wl = dataclasses.replace(ri.qwen_qk(4096), neox=neox)
    want = oracle.run_qk_norm_rope(wl)
    for variant in ("auto", "direct"):
        check(wl, variant, want)


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("variant", VARIANTS)
def test_head_dims_and_dtypes(head_dim, dtype, variant):
    for neox in (True, False):
        check(ri.make_qk_workload(f"qk_{head_dim}_{dtype}", 397, 6, 2, head_dim, dtype=dtype, neox=neox,
                                  sigma=3.0, seed=head_dim), variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_edge_cases(variant):
    check(ri.make_qk_workload("qk_one", 1, 8, 1, 128, seed=2), variant)
    check(ri.make_qk_workload("qk_noq", 33, 0, 3, 128, seed=3), variant)
    check(ri.make_qk_workload("qk_nokv", 33, 5, 0, 128, seed=4), variant)
    wl = ri.make_qk_workload("qk_range", 350, 4, 2, 128, max_pos=32, seed=5)
    wl.positions[[3, 17, 49, 200, 349]] = [32, -1, 1 << 40, -(1 << 40), 31]
    check(wl, variant)


@pytest.mark.parametrize("variant", VARIANTS)
def test_head_counts(variant):
    """Head groups per token above the pipelined form's 16 warps (D = 256:
    two heads per warp, 36 heads), a ragged last group, many heads of
    D = 64, and a token too large for two ring stages (the pipelined request
    runs as the warp kernel)."""
    check(ri.make_qk_workload("qk_18groups", 301, 32, 4, 256, seed=6), variant)
    check(ri.make_qk_workload("qk_ragged", 211, 7, 2, 128, neox=False, seed=7), variant)
    check(ri.make_qk_workload("qk_d64", 257, 64, 8, 64, seed=8), variant)
    check(ri.make_qk_workload("qk_huge", 9, 200, 20, 256, seed=9), variant)


def test_argument_errors():
    wl = ri.make_qk_workload("qk_err", 4, 2, 1, 128)
    qkv = P.dev_act(wl.qkv, wl.dtype)
    pos = torch.from_numpy(wl.positions).cuda()
    cs = torch.from_numpy(wl.cos_sin).cuda()
    w = P.dev_act(wl.q_weight, wl.dtype)
    with pytest.raises(rq.RmsqError) as ei:
        rq.qk_norm_rope(qkv, pos, cs, w, w, 1e-6, 2, 1, 96)        # head_dim 96 not supported
    assert ei.value.status == rq.ERR_UNSUPPORTED_SHAPE
    with pytest.raises(rq.RmsqError) as ei:
        rq.qk_norm_rope(qkv, pos, cs, w, w, -1.0, 2, 1, 128)
    assert ei.value.status == rq.ERR_INVALID_ARG
