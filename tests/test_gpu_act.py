"""SiLU+Mul + quantisation on the GPU against the oracle, bit for bit.

Same bar as the norm op: codes and scales identical (the CUDA path evaluates
e^x, the division and the products in the oracle's binary32 steps).
"""
import numpy as np
import pytest
import torch

import _parity as P
import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu
MODES = ["fp8_static", "fp8_per_token", "fp8_group128_row", "fp8_group128_col", "fp8_group64_row",
         "fp8_group64_col", "nvfp4"]


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def run_gpu(wl, mode, scale_in):
    gu = P.dev_act(wl.gate_up, wl.dtype)
    s = torch.tensor([scale_in or 0.0], dtype=torch.float32, device="cuda")
    q, sc = rq.silu_mul_quant(gu, mode, s)
    torch.cuda.synchronize()
    return {"q": q.cpu().numpy(), "scales": None if sc is None else sc.cpu().numpy(), "residual_out": None}


def check(wl, mode, nthreads=8):
    want = oracle.run_silu_mul_workload(wl, mode, nthreads=nthreads)
    got = run_gpu(wl, mode, want["scale_in"])
    return P.compare(got, want, mode, f"{wl.name}/{mode}")


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_modes_and_dtypes(mode, dtype):
    for n, d in ((300, 2048), (3, 512), (1, 128)):
        check(ri.make_act_workload(f"act_{n}x{d}_{dtype}", n, d, dtype=dtype, seed=n + d), mode)


@pytest.mark.parametrize("d", [8, 24, 1000, 4104, 8200, 16400, 32768])
def test_ragged_and_wide_rows(d):
    """Every thread-per-row width (one to eight chunks per thread), ragged last warps."""
    mode = "fp8_per_token"
    check(ri.make_act_workload(f"act_7x{d}", 7, d, seed=d), mode)
    check(ri.make_act_workload(f"act_7x{d}", 7, d, seed=d), "fp8_static")


def test_extreme_gate_range():
    """Gates from -120 to 100: e^-g overflows to inf (silu = -0), underflows to
    0 and passes through the subnormal range; results still bit-exact."""
    for mode in ("fp8_per_token", "fp8_group128_row", "nvfp4"):
        wl = ri.make_act_workload("act_range", 64, 1024, gate_range=(-120.0, 100.0), seed=21)
        check(wl, mode)


@pytest.mark.parametrize("mode", ["fp8_group128_row", "fp8_static", "nvfp4"])
def test_llama_mlp_full_size(mode):
    """4096 tokens x d = 14336 (gate_up 4096 x 28672 bf16): every element."""
    check(ri.llama_mlp(4096), mode, nthreads=16)


def test_empty_and_errors():
    gu = torch.zeros(0, 256, dtype=torch.bfloat16, device="cuda")
    q, sc = rq.silu_mul_quant(gu, "fp8_per_token")
    assert q.shape == (0, 128)
    gu = torch.zeros(4, 2 * 100, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rq.RmsqError) as ei:
        rq.silu_mul_quant(gu, "fp8_group128_row")    # d = 100 not a multiple of 128
    assert ei.value.status == rq.ERR_UNSUPPORTED_SHAPE
    big = torch.zeros(1, 2 * 32776, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(rq.RmsqError) as ei:
        rq.silu_mul_quant(big, "fp8_per_token")
    assert ei.value.status == rq.ERR_UNSUPPORTED_SHAPE


def _all_bf16_values():
    v = (np.arange(65536, dtype=np.uint32) << 16).view(np.float32)
    return v[np.isfinite(v)]


@pytest.mark.parametrize("kind", ["exp", "exp_mid", "silu"])
def test_activation_steps_on_every_bf16_input(kind):
    """The GPU's e^x (both step sequences) and silu against the oracle's on all
    finite bf16 values (and their negations, for e^-g), element by element."""
    x = _all_bf16_values()
    x = np.concatenate([x, -x]).astype(np.float32)
    if kind == "exp_mid":
        x = x[np.abs(x) <= 87.0]
    got = rq.debug_activation(kind, torch.from_numpy(x).cuda()).cpu().numpy()
    want = oracle.expf(x) if kind.startswith("exp") else oracle.silu(x)
    bad = got.view(np.uint32) != want.view(np.uint32)
    bad &= ~(np.isnan(got) & np.isnan(want))
    assert not bad.any(), (int(bad.sum()), x[bad][:8].tolist(), got[bad][:8].tolist(), want[bad][:8].tolist())


def test_silu_mul_on_random_pairs():
    rng = np.random.default_rng(1)
    g = rng.normal(0, 3, 2_000_003).astype(np.float32)
    u = rng.normal(0, 1, g.size).astype(np.float32)
    got = rq.debug_activation("silu_mul", torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda()).cpu().numpy()
    want = (oracle.silu(g) * u).astype(np.float32)
    bad = got.view(np.uint32) != want.view(np.uint32)
    assert not bad.any(), (int(bad.sum()), g[bad][:8].tolist(), got[bad][:8].tolist(), want[bad][:8].tolist())
