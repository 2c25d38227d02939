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


def run_gpu(wl):
    qkv = P.dev_act(wl.qkv, wl.dtype)
    pos = torch.from_numpy(wl.positions).cuda()
    cs = torch.from_numpy(wl.cos_sin).cuda()
    qw, kw = P.dev_act(wl.q_weight, wl.dtype), P.dev_act(wl.k_weight, wl.dtype)
    rq.qk_norm_rope(qkv, pos, cs, qw, kw, wl.eps, wl.nq, wl.nkv, wl.head_dim, wl.neox)
    torch.cuda.synchronize()
    return P.host_bits(qkv)


def check(wl):
    want = oracle.run_qk_norm_rope(wl)
    got = run_gpu(wl)
    bad = np.count_nonzero(got != want)
    assert bad == 0, f"{wl.name}: {bad} of {want.size} elements differ"


@pytest.mark.parametrize("neox", [True, False], ids=["neox", "gptj"])
def test_qwen_attention_shape(neox):
    """4096 tokens, 32 q heads, 4 kv heads, head_dim 128 (Qwen3-30B-A3B)."""
    check(dataclasses.replace(ri.qwen_qk(4096), neox=neox))


@pytest.mark.parametrize("head_dim", [64, 128, 256])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_head_dims_and_dtypes(head_dim, dtype):
    for neox in (True, False):
        check(ri.make_qk_workload(f"qk_{head_dim}_{dtype}", 97, 6, 2, head_dim, dtype=dtype, neox=neox,
                                  sigma=3.0, seed=head_dim))


def test_edge_cases():
    check(ri.make_qk_workload("qk_one", 1, 8, 1, 128, seed=2))
    check(ri.make_qk_workload("qk_noq", 33, 0, 3, 128, seed=3))
    check(ri.make_qk_workload("qk_nokv", 33, 5, 0, 128, seed=4))
    wl = ri.make_qk_workload("qk_range", 50, 4, 2, 128, max_pos=32, seed=5)
    wl.positions[[3, 17, 49]] = [32, -1, 1 << 40]
    check(wl)


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
