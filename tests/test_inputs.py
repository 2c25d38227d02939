"""The seeded input generators: deterministic, and shaped like the stated workloads."""
import numpy as np
import torch

import rmsq_inputs as ri


def test_streams_are_deterministic_and_distinct():
    a = ri.uniform(0, 1, 1000)
    assert np.array_equal(a, ri.uniform(0, 1, 1000))
    assert not np.array_equal(a, ri.uniform(0, 2, 1000))
    assert not np.array_equal(a, ri.uniform(1, 1, 1000))
    # prefix property of a counter-based stream
    assert np.array_equal(ri.uniform(0, 1, 10), a[:10])
    assert a.min() >= 0 and a.max() < 1


def test_normal_moments():
    z = ri.normal(0, 1, 1 << 20)
    assert abs(z.mean()) < 5e-3 and abs(z.std() - 1) < 5e-3


def test_student_t3_tails():
    t = ri.student_t3(0, 1, 1 << 18)
    # P(|T3| > 5) = 0.0154 for 3 degrees of freedom
    frac = np.mean(np.abs(t) > 5)
    assert 0.012 < frac < 0.019


def test_llama_workload_shape_and_scale():
    wl = ri.llama(n_tokens=64)
    assert wl.x.shape == (64, 4096) and wl.residual.shape == (64, 4096)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).float()
    r = torch.from_numpy(wl.residual.view(np.int16)).view(torch.bfloat16).float()
    assert abs(x.std().item() - 1) < 0.02 and abs(r.std().item() - 2) < 0.04
    w = torch.from_numpy(wl.weight.view(np.int16)).view(torch.bfloat16).float()
    assert abs(w.mean().item() - 1) < 0.01 and abs(w.std().item() - 0.1) < 0.01


def test_dsv3_outlier_channels():
    wl = ri.dsv3(n_tokens=16)
    ch = wl.meta["outlier_channels"]
    assert len(ch) == 72 and len(set(ch)) == 72
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.bfloat16).float()
    mask = np.zeros(7168, bool)
    mask[ch] = True
    assert x[:, mask].std() > 15 and x[:, ~mask].std() < 1.1


def test_decode_workload_is_finite_fp16():
    wl = ri.decode(n_tokens=256)
    x = torch.from_numpy(wl.x.view(np.int16)).view(torch.float16).float()
    r = torch.from_numpy(wl.residual.view(np.int16)).view(torch.float16).float()
    assert torch.isfinite(x + r).all() and (x + r).abs().max() < 65504
    assert len(wl.meta["outlier_channels"]) == 8
