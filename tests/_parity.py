"""Helpers for the GPU-vs-oracle parity tests: upload seeded inputs, run both
sides, compare element by element.

Bar (the stated tolerance of the path): residual_out and scales bit-exact;
quantised codes bit-exact except at most 1 code step on at most 1e-4 of the
elements.  The CUDA path is designed to be bit-exact everywhere, so the
mismatch counts are reported and the tests also require them to be zero.
Every check runs both kernel variants (direct and pipelined) on the same
inputs.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq

MAX_MISMATCH_FRAC = 1e-4
MAX_STEP = 1
VARIANTS = ("direct", "pipelined")
_TDT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def dev_act(bits: np.ndarray, dtype: str, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(_TDT[dtype]).to(device)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def run_gpu(wl, mode: str, scale_in: float | None, *, in_place: bool = False, stream=None,
            variant: str = "auto"):
    x = dev_act(wl.x, wl.dtype)
    r = None if wl.residual is None else dev_act(wl.residual, wl.dtype)
    w = dev_act(wl.weight, wl.dtype)
    s = torch.tensor([scale_in if scale_in is not None else 0.0], dtype=torch.float32, device="cuda")
    q, sc, ro = rq.fused_add_rmsnorm_quant(x, r, w, wl.eps, mode, s,
                                           residual_out=r if (in_place and r is not None) else None,
                                           stream=stream, variant=variant)
    torch.cuda.synchronize()
    assert rq.take_fault_flags() == 0, "a pipelined CTA gave up waiting for its copies"
    return {"q": q.cpu().numpy(), "scales": None if sc is None else sc.cpu().numpy(),
            "residual_out": None if ro is None else host_bits(ro)}


def code_steps(got: np.ndarray, want: np.ndarray, mode: str) -> np.ndarray:
    """Per-element code distance (sign-magnitude), FP8 bytes or E2M1 nibbles."""
    if mode == "nvfp4":
        g = np.stack([got & 0xF, got >> 4], -1).astype(np.int32)
        w = np.stack([want & 0xF, want >> 4], -1).astype(np.int32)
        sg, sw, mg, mw = g >> 3, w >> 3, g & 7, w & 7
    else:
        g, w = got.astype(np.int32), want.astype(np.int32)
        sg, sw, mg, mw = g >> 7, w >> 7, g & 0x7F, w & 0x7F
    same = sg == sw
    return np.where(same, np.abs(mg - mw), mg + mw)


def compare(got: dict, want: dict, mode: str, label: str = "") -> dict:
    """Assert the parity bar; return the mismatch report."""
    if want["residual_out"] is not None:
        assert got["residual_out"] is not None
        bad = np.count_nonzero(got["residual_out"] != want["residual_out"])
        assert bad == 0, f"{label}: residual_out differs in {bad} elements"
    if want["scales"] is not None:
        g, w = got["scales"], want["scales"]
        assert g.shape == w.shape, (g.shape, w.shape)
        gb = g.view(np.uint32) if g.dtype == np.float32 else g
        wb = w.view(np.uint32) if w.dtype == np.float32 else w
        bad = np.count_nonzero(gb != wb)
        assert bad == 0, f"{label}: {bad} of {w.size} scales differ"
    assert got["q"].shape == want["q"].shape
    steps = code_steps(got["q"], want["q"], mode)
    n_bad = int(np.count_nonzero(steps))
    frac = n_bad / max(1, steps.size)
    mx = int(steps.max()) if steps.size else 0
    report = {"label": label, "elements": int(steps.size), "mismatches": n_bad,
              "fraction": frac, "max_step": mx}
    print(f"parity {label}: {report}")
    assert frac <= MAX_MISMATCH_FRAC and mx <= MAX_STEP, f"{label}: {report}"
    assert n_bad == 0, f"{label}: codes not bit-exact: {report}"
    return report


def check(wl, mode: str, *, scale_in: float | None = None, nthreads: int = 8,
          in_place: bool = False, label: str | None = None, variants=VARIANTS) -> list:
    want = oracle.run_workload(wl, mode, scale_in=scale_in, nthreads=nthreads)
    reports = []
    for v in variants:
        got = run_gpu(wl, mode, want["scale_in"], in_place=in_place, variant=v)
        reports.append(compare(got, want, mode, f"{label or wl.name + '/' + mode}/{v}"))
    return reports
