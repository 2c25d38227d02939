"""The library's hardware E4M3 / E2M1 conversions against the oracle's encoders.

Inputs: every fp32 bit pattern within 64 ulps of each code value and of each
midpoint between neighbouring codes (both signs), 16M random bit patterns
spread over the relevant binades, and the special values.  This pins rounding
(nearest even), saturation, signed zero and the nibble placement that every
kernel relies on.
"""
import numpy as np
import pytest
import torch

import oracle
import residual_add_rmsnorm_rmsq_gb300 as rq
from rmsq_inputs import uniform

pytestmark = pytest.mark.gpu


def _neighbourhoods(points: np.ndarray, width: int = 64) -> np.ndarray:
    pts = np.abs(points.astype(np.float32)).view(np.uint32).astype(np.int64)
    offs = np.arange(-width, width + 1, dtype=np.int64)
    bits = (pts[:, None] + offs[None, :]).ravel()
    bits = bits[(bits >= 0) & (bits < 0x7F800000)].astype(np.uint32)
    pos = bits.view(np.float32)
    return np.concatenate([pos, -pos])


def _inputs(values: np.ndarray, extra_random: int, seed: int, lo_exp: int, hi_exp: int) -> np.ndarray:
    mids = (values[:-1].astype(np.float64) + values[1:]) / 2
    pts = np.concatenate([values, mids.astype(np.float32)])
    u = uniform(seed, 1, 2 * extra_random)
    mag = 2.0 ** (lo_exp + (hi_exp - lo_exp) * u[:extra_random])
    rnd = np.where(u[extra_random:] < 0.5, -mag, mag).astype(np.float32)
    special = np.array([0.0, -0.0, np.inf, -np.inf, 1e-45, -1e-45, 3.4e38, -3.4e38], np.float32)
    return np.concatenate([_neighbourhoods(pts), rnd, special]).astype(np.float32)


def _run(kind: str, v: np.ndarray) -> np.ndarray:
    out = rq.debug_convert(kind, torch.from_numpy(v).cuda())
    torch.cuda.synchronize()
    return out.cpu().numpy()


def test_e4m3_conversion_matches_oracle(rmsq_gpu):
    table = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    v = _inputs(table, 1 << 24, 41, -16, 10)
    v = np.concatenate([v, np.array([np.nan, -np.nan], np.float32)])
    got, want = _run("e4m3", v), oracle.e4m3_encode(v)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]


def test_e2m1_conversion_matches_oracle(rmsq_gpu):
    table = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)
    v = _inputs(table, 1 << 22, 42, -8, 4)
    got, want = _run("e2m1", v), oracle.e2m1_encode(v)
    bad = np.flatnonzero(got != want)
    assert bad.size == 0, [(float(v[i]), hex(got[i]), hex(want[i])) for i in bad[:10]]
