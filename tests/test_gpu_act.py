"""SiLU+Mul + quantisation on the GPU against the oracle.

The oracle takes silu from its plain definition (binary64, rounded once); the
CUDA path evaluates e^x, the sum and the division in binary32 steps, so its
activation a = silu(g) * u can sit a few ulps from the oracle's.  Two checks,
therefore, on every workload:

1. exactness of the quantisation: the kernel's codes and scales equal the
   oracle's quantisation step applied to the kernel's own activations (read
   back through the library's elementwise debug entry), bit for bit;
2. the bar against the independent oracle: codes within one step on at most
   1e-4 of the elements, every scale within ACT_SCALE_ULP binary32 ulps of
   the oracle's (a per-token / group scale moves only when its amax element's
   activation does); both counts are printed.

ACT_SCALE_ULP follows from the arithmetic: the kernel's e^x is within
2.4 ulp (4.8 * 2^-24 relative: the hardware 2^x's two ulps and the rounding
of the reduced argument; EXP_ULP checks it on every bf16 input), 1 + e^-g
rounds once (2^-24), the approximate reciprocal is within one ulp
(2 * 2^-24) and the product g * r rounds once (2^-24), so its silu is within
8.8 * 2^-24 of the exact value; the oracle's is within 2^-24; both products
with u round once more (2^-24 each).  The two activations are therefore
within 11.8 * 2^-24 relative, at most 11.8 ulps, and the scale's own
rounding adds at most one.
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
ACT_SCALE_ULP = 13
EXP_ULP = 2.5           # the kernel's e^x: Cody-Waite reduction + the hardware 2^x
SILU_ULP = 9.0          # its silu: e^x, 1 + e^-g, the approximate reciprocal, the product


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def run_gpu(wl, mode, scale_in):
    gu = P.dev_act(wl.gate_up, wl.dtype)
    s = torch.tensor([scale_in or 0.0], dtype=torch.float32, device="cuda")
    q, sc = rq.silu_mul_quant(gu, mode, s)
    torch.cuda.synchronize()
    return {"q": q.cpu().numpy(), "scales": None if sc is None else sc.cpu().numpy(), "residual_out": None}


def kernel_activations(wl):
    """The kernel's own a = silu(g) * u, elementwise on the device."""
    gu = P.dev_act(wl.gate_up, wl.dtype).float()
    d = wl.d
    a = rq.debug_activation("silu_mul", gu[:, :d].contiguous(), gu[:, d:].contiguous())
    torch.cuda.synchronize()
    return a.cpu().numpy()


def _ulps(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Distance in binary32 ulps between positive floats (their bit patterns)."""
    return np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))


def check(wl, mode, nthreads=8):
    want = oracle.run_silu_mul_workload(wl, mode, nthreads=nthreads)
    got = run_gpu(wl, mode, want["scale_in"])
    label = f"{wl.name}/{mode}"
    # 1. the quantisation of the kernel's own activations, bit for bit
    mine = oracle.run_quant_f32(kernel_activations(wl), mode=mode, scale_in=want["scale_in"] or 0.0,
                                nthreads=nthreads)
    assert np.array_equal(got["q"], mine["q"]), f"{label}: codes differ from the quantisation of the kernel's a"
    if mine["scales"] is not None:
        assert np.array_equal(got["scales"].view(np.uint8), mine["scales"].view(np.uint8)), label
    # 2. against the independent oracle
    steps = P.code_steps(got["q"], want["q"], mode)
    n_bad = int(np.count_nonzero(steps))
    report = {"label": label, "elements": int(steps.size), "mismatches": n_bad,
              "fraction": n_bad / max(1, steps.size), "max_step": int(steps.max()) if steps.size else 0}
    if want["scales"] is not None:
        g, w = got["scales"], want["scales"]
        if g.dtype == np.float32:
            d_ulp = _ulps(g, w)
            report["scales"] = int(g.size)
            report["scale_mismatches"] = int(np.count_nonzero(d_ulp))
            report["scale_max_ulp"] = int(d_ulp.max()) if d_ulp.size else 0
            assert report["scale_max_ulp"] <= ACT_SCALE_ULP, report
        else:   # NVFP4 block scales: E4M3 codes of amax / 6 * gs
            sd = P.code_steps(g, w, "fp8_static")
            report["scale_mismatches"] = int(np.count_nonzero(sd))
            assert int(sd.max()) <= 1 and np.count_nonzero(sd) <= max(1, P.MAX_MISMATCH_FRAC * sd.size), report
    print(f"parity {report}")
    assert report["fraction"] <= P.MAX_MISMATCH_FRAC and report["max_step"] <= P.MAX_STEP, report
    return report


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
    0 and passes through the subnormal range; results still within the bar."""
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
    """The GPU's e^x (both step sequences) and silu on all finite bf16 values
    (and their negations, for e^-g), against the double-precision
    definitions, within the bounds of their binary32 steps."""
    x = _all_bf16_values()
    x = np.concatenate([x, -x]).astype(np.float32)
    if kind == "exp_mid":
        x = x[np.abs(x) <= 87.0]
    got = rq.debug_activation(kind, torch.from_numpy(x).cuda()).cpu().numpy().astype(np.float64)
    x64 = x.astype(np.float64)
    with np.errstate(over="ignore"):
        want = np.exp(x64) if kind.startswith("exp") else x64 / (1.0 + np.exp(-x64))
    fin = np.isfinite(want) & (np.abs(want) >= 2.0 ** -126) & (np.abs(want) <= 3.0e38)
    if kind == "silu":
        # below g = -88.72 (ln of the largest binary32), e^-g overflows and the
        # kernel's silu is -0, where the exact value is below 2^-120 in
        # magnitude (it quantises to a zero code under any scale the 1e-12
        # floor allows)
        flushed = (x64 < -88.5) & (got == 0.0)
        assert np.all(np.abs(want[flushed]) < 2.0 ** -120)
        assert np.all(flushed[x64 < -88.73])
        fin &= ~flushed
    sp = np.spacing(np.abs(want[fin]).astype(np.float32)).astype(np.float64)
    err = np.abs(got[fin] - want[fin]) / sp
    bound = EXP_ULP if kind.startswith("exp") else SILU_ULP
    assert err.max() <= bound, (err.max(), x[fin][np.argmax(err)])
    # outside the normal range: overflow to inf, underflow to (signed) zero
    big = np.isfinite(x64) & ~np.isfinite(want)
    assert np.all(np.isinf(got[big]))
    tiny = np.abs(want) < 2.0 ** -151        # well below half the smallest subnormal
    assert np.all(got[tiny] == 0.0)


def test_silu_mul_on_random_pairs():
    """silu(g) * u from the debug entry: within the activation bound of the
    double-precision product."""
    rng = np.random.default_rng(1)
    g = rng.normal(0, 3, 2_000_003).astype(np.float32)
    u = rng.normal(0, 1, g.size).astype(np.float32)
    got = rq.debug_activation("silu_mul", torch.from_numpy(g).cuda(), torch.from_numpy(u).cuda()).cpu().numpy()
    g64 = g.astype(np.float64)
    want = g64 / (1.0 + np.exp(-g64)) * u.astype(np.float64)
    ok = np.abs(want) > 1e-30
    sp = np.spacing(np.abs(want[ok]).astype(np.float32)).astype(np.float64)
    err = np.abs(got[ok].astype(np.float64) - want[ok]) / sp
    assert err.max() <= SILU_ULP + 1.0, err.max()
