"""Pins of the oracle's number formats against things other than itself.

E4M3 decode is checked against torch.float8_e4m3fn; E4M3 / E2M1 encode against
a brute-force nearest-code search over the decoded tables (ties to the even
code, saturation at the largest finite value); bf16 / fp16 rounding against
torch and numpy conversions.  The formats are the OCP FP8 E4M3 and FP4 E2M1
ones that the NVFP4 and FP8 schemes of the pages name (vLLM docs "Fusion
torch.compile passes", support matrix; vLLM PR #51925 summary).
"""
import numpy as np
import pytest
import torch

from rmsq_inputs import uniform


def _brute_nearest(vals: np.ndarray, table: np.ndarray, sign_bit: int) -> np.ndarray:
    """Nearest entry of the non-negative, increasing ``table`` to |v| (ties to
    the even index), with the sign bit of v set in the result."""
    a = np.abs(vals.astype(np.float64))
    d = np.abs(a[:, None] - table[None, :].astype(np.float64))
    best = d.min(axis=1, keepdims=True)
    cand = d == best
    idx = np.arange(table.size)[None, :]
    even = np.where(cand & (idx % 2 == 0), idx, 10 ** 6).min(axis=1)
    anyc = np.where(cand, idx, 10 ** 6).min(axis=1)
    ncand = cand.sum(axis=1)
    code = np.where(ncand > 1, even, anyc).astype(np.uint8)
    return code | np.where(np.signbit(vals), sign_bit, 0).astype(np.uint8)


def _e4m3_table(orc):
    return orc.e4m3_decode(np.arange(0x7f, dtype=np.uint8))   # 0x00 .. 0x7e


def test_e4m3_decode_matches_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert nan.sum() == 2 and ours[0x7e] == 448.0 and ours[0x01] == 2.0 ** -9


def test_e4m3_roundtrip_every_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7f, 0xff)], np.uint8)
    assert np.array_equal(orc.e4m3_encode(orc.e4m3_decode(codes)), codes)


def test_e4m3_midpoints_tie_to_even(orc):
    table = _e4m3_table(orc)
    for c in range(0x7e):
        lo, hi = np.float32(table[c]), np.float32(table[c + 1])
        mid = np.float32((np.float64(lo) + np.float64(hi)) / 2)      # exact in fp32
        assert np.float64(mid) == (np.float64(lo) + np.float64(hi)) / 2
        even = c if c % 2 == 0 else c + 1
        got = orc.e4m3_encode(np.array([mid, -mid, np.nextafter(mid, np.float32(0)),
                                        np.nextafter(mid, np.float32(1e9))], np.float32))
        assert list(got) == [even, even | 0x80, c, c + 1], hex(c)


def test_e4m3_saturation_and_specials(orc):
    v = np.array([448, 449, 463.99, 464, 480, 1e30, np.inf, -448, -1e30, -np.inf, np.nan,
                  0.0, -0.0, 2.0 ** -10, 2.0 ** -10 * 1.0000001, -1e-30], np.float32)
    expect = [0x7e, 0x7e, 0x7e, 0x7e, 0x7e, 0x7e, 0x7e, 0xfe, 0xfe, 0xfe, 0x7f,
              0x00, 0x80, 0x00, 0x01, 0x80]
    assert list(orc.e4m3_encode(v)) == expect


def test_e4m3_encode_brute_force(orc):
    table = _e4m3_table(orc)
    u = uniform(11, 1, 300000)
    lin = (u[:100000] * 2 - 1) * 500.0                                  # linear in [-500, 500]
    log = np.sign(u[100000:200000] - 0.5) * 2.0 ** (-14 + 24 * u[200000:])  # 2^-14 .. 2^10
    vals = np.concatenate([lin, log]).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), _brute_nearest(vals, table, 0x80))


def test_e4m3_encode_matches_torch_in_range(orc):
    u = uniform(12, 1, 200000)
    vals = ((u * 2 - 1) * 448.0).astype(np.float32)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(orc.e4m3_encode(vals), ref)


E2M1_VALUES = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6], np.float32)


def test_e2m1_decode_table(orc):
    codes = np.arange(16, dtype=np.uint8)
    dec = orc.e2m1_decode(codes)
    assert np.array_equal(dec[:8], E2M1_VALUES)
    assert np.array_equal(dec[8:], -E2M1_VALUES) and np.signbit(dec[8])


def test_e2m1_worked_values(orc):
    # ties: 0.25 -> 0, 0.75 -> 1, 1.25 -> 1, 1.75 -> 2, 2.5 -> 2, 3.5 -> 4, 5 -> 4; 7 saturates
    v = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 7.0, -0.0, -0.2, -6.5, np.inf], np.float32)
    assert list(orc.e2m1_encode(v)) == [0, 2, 2, 4, 4, 6, 6, 7, 8, 8, 15, 7]


def test_e2m1_encode_brute_force(orc):
    u = uniform(13, 1, 200000)
    vals = ((u * 2 - 1) * 8.0).astype(np.float32)
    mids = (E2M1_VALUES[:-1] + E2M1_VALUES[1:]) / 2
    vals = np.concatenate([vals, mids, -mids, np.nextafter(mids, np.float32(0)),
                           np.nextafter(mids, np.float32(9))]).astype(np.float32)
    assert np.array_equal(orc.e2m1_encode(vals), _brute_nearest(vals, E2M1_VALUES, 0x8))


def test_bf16_rounding_matches_torch(orc):
    u = uniform(14, 1, 400000)
    bits = (u * 2 ** 32).astype(np.uint64).astype(np.uint32)
    vals = bits.view(np.float32)
    vals = vals[np.isfinite(vals)]
    # exact halfway cases: low 16 bits 0x8000 with both parities of bit 16
    half = ((bits[:1000] & 0xFFFF0000) | 0x8000).view(np.float32)
    vals = np.concatenate([vals, half[np.isfinite(half)],
                           np.array([3.3895314e38, 3.4028235e38, 1e-40, -1e-45], np.float32)])
    ref = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.float_to_act(vals, "bf16"), ref)


def test_fp16_rounding_matches_numpy(orc):
    u = uniform(15, 1, 400000)
    vals = (np.sign(u[:200000] - 0.5) * 2.0 ** (-30 + 48 * u[200000:])).astype(np.float32)
    table = np.arange(0, 0x7c00, dtype=np.uint16).view(np.float16).astype(np.float32)
    mids = ((table[:-1].astype(np.float64) + table[1:]) / 2).astype(np.float32)
    extra = np.array([65504, 65519.99, 65520, 70000, np.inf, -np.inf, 0.0, -0.0], np.float32)
    vals = np.concatenate([vals, mids, -mids, extra])
    ref = vals.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.float_to_act(vals, "fp16"), ref)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_widening_every_pattern(orc, dtype):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.act_to_float(bits, dtype)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    ref = torch.from_numpy(bits.view(np.int16)).view(tdt).float().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan].view(np.uint32), ref[~nan].view(np.uint32))
