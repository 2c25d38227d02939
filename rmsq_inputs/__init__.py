"""Seeded synthetic inputs for the fused residual-add + RMSNorm + quantisation path.

This module is shared by the CPU oracle side and the CUDA side of every test and
of the benchmark.  It only *draws* numbers; it holds none of the method's
arithmetic (no normalisation, no scales, no quantisation).

Random stream
-------------
Counter-based splitmix64: the i-th 64-bit word of stream ``k`` under seed ``s``
is ``mix64(key(s, k) + (i + 1) * 0x9E3779B97F4A7C15)`` (Steele, Lea, Flood,
"Fast splittable pseudorandom number generators", OOPSLA 2014).  Uniforms take
the top 53 bits; normals come from the Box-Muller transform on consecutive
uniform pairs; Student-t(3) is ``Z / sqrt(chi2_3 / 3)`` with ``chi2_3`` the sum
of three squared normals.  Values are drawn in float64, rounded to float32 and
then to the activation type (bf16 or fp16) with round-to-nearest-even
(``torch.Tensor.to``).  The same host bytes feed the oracle and the GPU.

Workloads
---------
The shapes and value distributions follow the workloads of the pages (the
Llama-, DeepSeek-V3- and Qwen3-shaped layers the fusion is used on); every
tensor stream uses seed 0 unless a test asks otherwise.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_CHUNK = 1 << 22

# stream ids: one independent stream per tensor / purpose
STREAM_X, STREAM_RES, STREAM_W, STREAM_OUTLIER, STREAM_AUX = 1, 2, 3, 4, 5
STREAM_GATE, STREAM_UP = 6, 7
STREAM_QKV, STREAM_POS = 8, 9


def _mix64(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def _key(seed: int, stream: int) -> np.uint64:
    with np.errstate(over="ignore"):
        a = np.array([(seed * 0x632BE59BD9B4E019 + stream * 0x8CB92BA72F3D8DD7) & (2**64 - 1)],
                     dtype=np.uint64)
        return _mix64(a)[0]


def uniform(seed: int, stream: int, n: int) -> np.ndarray:
    """n float64 uniforms in [0, 1) from stream ``stream`` of ``seed``."""
    out = np.empty(n, dtype=np.float64)
    key = _key(seed, stream)
    with np.errstate(over="ignore"):
        for s in range(0, n, _CHUNK):
            e = min(n, s + _CHUNK)
            idx = np.arange(s + 1, e + 1, dtype=np.uint64)
            z = _mix64(key + idx * _GAMMA)
            out[s:e] = (z >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)
    return out


def normal(seed: int, stream: int, n: int) -> np.ndarray:
    """n standard normals (float64) by Box-Muller on consecutive uniform pairs."""
    m = (n + 1) // 2
    u = uniform(seed, stream, 2 * m)
    u1, u2 = u[0::2], u[1::2]
    rad = np.sqrt(-2.0 * np.log1p(-u1))
    ang = 2.0 * math.pi * u2
    z = np.empty(2 * m, dtype=np.float64)
    z[0::2] = rad * np.cos(ang)
    z[1::2] = rad * np.sin(ang)
    return z[:n]


def student_t3(seed: int, stream: int, n: int) -> np.ndarray:
    """n Student-t(df=3) draws: Z / sqrt((Z1^2 + Z2^2 + Z3^2) / 3), float64."""
    z = normal(seed, stream, 4 * n).reshape(n, 4)
    chi2 = z[:, 1] ** 2 + z[:, 2] ** 2 + z[:, 3] ** 2
    return z[:, 0] / np.sqrt(chi2 / 3.0)


def pick_channels(seed: int, stream: int, hidden: int, k: int) -> np.ndarray:
    """k distinct channel indices by a seeded partial Fisher-Yates shuffle."""
    perm = np.arange(hidden)
    u = uniform(seed, stream, k)
    for i in range(k):
        j = i + int(u[i] * (hidden - i))
        perm[i], perm[j] = perm[j], perm[i]
    return np.sort(perm[:k])


_TORCH_DT = {"bf16": torch.bfloat16, "fp16": torch.float16}


def to_bits(values: np.ndarray, dtype: str) -> np.ndarray:
    """float64 -> float32 (RNE) -> bf16/fp16 (RNE); returns the uint16 bit patterns."""
    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32)).to(_TORCH_DT[dtype])
    return t.view(torch.int16).numpy().view(np.uint16).copy()


@dataclass
class Workload:
    """One synthetic problem: bit patterns of x, residual (or None), weight."""
    name: str
    n_tokens: int
    hidden: int
    dtype: str                  # "bf16" | "fp16"
    eps: float
    x: np.ndarray               # uint16 [n, H]
    residual: np.ndarray | None  # uint16 [n, H] or None
    weight: np.ndarray          # uint16 [H]
    static_scale: float | None = None
    meta: dict = field(default_factory=dict)


def make_workload(name: str, n_tokens: int, hidden: int, *, dtype: str = "bf16",
                  dist: str = "normal", x_sigma: float = 1.0, res_sigma: float = 1.0,
                  residual: bool = True, n_outliers: int = 0, outlier_mult: float = 1.0,
                  t_clamp: float | None = None, eps: float = 1e-6,
                  static_scale: float | None = None, seed: int = 0) -> Workload:
    """Draw x, residual and weight for an [n_tokens, hidden] layer.

    dist "normal": x ~ x_sigma * N(0,1), residual ~ res_sigma * N(0,1).
    dist "t3": both ~ Student-t(3), clamped to |v| <= t_clamp when given.
    n_outliers channels (same channels in x and residual) are multiplied by
    outlier_mult.  weight = 1 + 0.1 * N(0,1).
    """
    n, H = int(n_tokens), int(hidden)
    cnt = n * H

    def draw(stream: int, sigma: float) -> np.ndarray:
        if dist == "normal":
            v = normal(seed, stream, cnt) * sigma
        elif dist == "t3":
            v = student_t3(seed, stream, cnt) * sigma
        else:
            raise ValueError(dist)
        if t_clamp is not None:
            np.clip(v, -t_clamp, t_clamp, out=v)
        return v.reshape(n, H)

    chans = pick_channels(seed, STREAM_OUTLIER, H, n_outliers) if n_outliers else np.zeros(0, int)
    xv = draw(STREAM_X, x_sigma)
    if len(chans):
        xv[:, chans] *= outlier_mult
    x = to_bits(xv, dtype).reshape(n, H)
    del xv
    r = None
    if residual:
        rv = draw(STREAM_RES, res_sigma)
        if len(chans):
            rv[:, chans] *= outlier_mult
        r = to_bits(rv, dtype).reshape(n, H)
        del rv
    w = to_bits(1.0 + 0.1 * normal(seed, STREAM_W, H), dtype)
    return Workload(name, n, H, dtype, float(eps), x, r, w, static_scale,
                    {"outlier_channels": chans.tolist(), "dist": dist})


# ----------------------------------------------------------------------------
# The five workloads of the scope table (sizes, distributions, eps, scales).
# ----------------------------------------------------------------------------

def pr1(seed: int = 0) -> Workload:
    """64 x 512 bf16, x, residual ~ N(0,1), eps 1e-6, FP8 static scale 0.05."""
    return make_workload("pr1_64x512", 64, 512, eps=1e-6, static_scale=0.05, seed=seed)


def llama(n_tokens: int = 4096, residual: bool = True, seed: int = 0) -> Workload:
    """Llama-8B-shaped: 4096 x 4096 bf16, x ~ N(0,1), residual ~ 2 N(0,1), eps 1e-5."""
    return make_workload(f"llama_{n_tokens}x4096", n_tokens, 4096, res_sigma=2.0,
                         residual=residual, eps=1e-5, seed=seed)


def dsv3(n_tokens: int = 8192, seed: int = 0) -> Workload:
    """DeepSeek-V3-shaped: 8192 x 7168 bf16 ~ N(0,1), 1 % of channels (72) x20, eps 1e-6."""
    H = 7168
    return make_workload(f"dsv3_{n_tokens}x{H}", n_tokens, H, n_outliers=round(0.01 * H),
                         outlier_mult=20.0, eps=1e-6, seed=seed)


def qwen_nvfp4(n_tokens: int = 4096, seed: int = 0) -> Workload:
    """Qwen3-30B-A3B-shaped: hidden 2048 bf16 ~ N(0,1), eps 1e-6 (NVFP4 layer)."""
    return make_workload(f"qwen_{n_tokens}x2048", n_tokens, 2048, eps=1e-6, seed=seed)


def decode(n_tokens: int = 1, residual: bool = True, seed: int = 0) -> Workload:
    """Decode sweep: fp16, hidden 8192, Student-t(3) clamped at 500, 8 channels x50, eps 1e-5."""
    return make_workload(f"decode_{n_tokens}x8192", n_tokens, 8192, dtype="fp16", dist="t3",
                         residual=residual, n_outliers=8, outlier_mult=50.0, t_clamp=500.0,
                         eps=1e-5, static_scale=0.1, seed=seed)


QWEN_TOKENS = (1, 16, 256, 4096, 16384)
DECODE_TOKENS = tuple(2 ** i for i in range(9))   # 1 .. 256


# ----------------------------------------------------------------------------
# SiLU+Mul + quantisation (the activation of a gated MLP).
# ----------------------------------------------------------------------------

@dataclass
class ActWorkload:
    """Bit patterns of one gated-MLP activation input: gate_up [n, 2d] holds
    the gate pre-activation in columns [0, d) and the up projection in
    [d, 2d) of every row."""
    name: str
    n_tokens: int
    d: int
    dtype: str
    gate_up: np.ndarray          # uint16 [n, 2d]
    static_scale: float | None = None


def make_act_workload(name: str, n_tokens: int, d: int, *, dtype: str = "bf16",
                      gate_sigma: float = 2.0, up_sigma: float = 1.0,
                      gate_range: tuple | None = None, static_scale: float | None = 0.05,
                      seed: int = 0) -> ActWorkload:
    """gate ~ gate_sigma * N(0,1) (or uniform on gate_range), up ~ up_sigma * N(0,1)."""
    n, d = int(n_tokens), int(d)
    if gate_range is None:
        g = normal(seed, STREAM_GATE, n * d) * gate_sigma
    else:
        lo, hi = gate_range
        g = lo + (hi - lo) * uniform(seed, STREAM_GATE, n * d)
    u = normal(seed, STREAM_UP, n * d) * up_sigma
    gu = np.empty((n, 2 * d), np.uint16)
    gu[:, :d] = to_bits(g, dtype).reshape(n, d)
    gu[:, d:] = to_bits(u, dtype).reshape(n, d)
    return ActWorkload(name, n, d, dtype, gu, static_scale)


def llama_mlp(n_tokens: int = 4096, seed: int = 0) -> ActWorkload:
    """Llama-8B-shaped MLP activation: d = 14336 (gate_up [n, 28672]) bf16."""
    return make_act_workload(f"llama_mlp_{n_tokens}x14336", n_tokens, 14336, seed=seed)


# ----------------------------------------------------------------------------
# QK-norm + RoPE (per-head RMSNorm of Q and K before the rotary embedding).
# ----------------------------------------------------------------------------

@dataclass
class QKWorkload:
    """qkv [n, (nq + 2 nkv) D] bit patterns (q heads, k heads, v heads per
    token), per-token positions, the fp32 cos / sin table [max_pos, D] (cos in
    the first D/2 columns, sin in the rest) and the q / k norm weights [D]."""
    name: str
    n_tokens: int
    nq: int
    nkv: int
    head_dim: int
    dtype: str
    eps: float
    neox: bool
    qkv: np.ndarray
    positions: np.ndarray
    cos_sin: np.ndarray
    q_weight: np.ndarray
    k_weight: np.ndarray


def rope_table(max_pos: int, head_dim: int, theta: float = 1e6) -> np.ndarray:
    """cos / sin of pos * theta^(-2i/D), i < D/2, computed in float64 and
    rounded to fp32 (an input of the op, like a model's cached table)."""
    half = head_dim // 2
    inv_freq = theta ** (-np.arange(half, dtype=np.float64) * 2.0 / head_dim)
    ang = np.arange(max_pos, dtype=np.float64)[:, None] * inv_freq[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def make_qk_workload(name: str, n_tokens: int, nq: int = 32, nkv: int = 4, head_dim: int = 128, *,
                     dtype: str = "bf16", neox: bool = True, max_pos: int = 8192, eps: float = 1e-6,
                     sigma: float = 1.0, seed: int = 0) -> QKWorkload:
    """qkv ~ sigma * N(0,1), positions uniform in [0, max_pos), weights 1 + 0.1 N(0,1)."""
    n, width = int(n_tokens), (nq + 2 * nkv) * head_dim
    qkv = to_bits(normal(seed, STREAM_QKV, n * width) * sigma, dtype).reshape(n, width)
    pos = np.minimum((uniform(seed, STREAM_POS, n) * max_pos).astype(np.int64), max_pos - 1)
    qw = to_bits(1.0 + 0.1 * normal(seed, STREAM_W, head_dim), dtype)
    kw = to_bits(1.0 + 0.1 * normal(seed, STREAM_AUX, head_dim), dtype)
    return QKWorkload(name, n, nq, nkv, head_dim, dtype, float(eps), neox, qkv, pos,
                      rope_table(max_pos, head_dim), qw, kw)


def qwen_qk(n_tokens: int = 4096, seed: int = 0) -> QKWorkload:
    """Qwen3-30B-A3B attention input: 32 q heads, 4 kv heads, head_dim 128, bf16, NeoX rotary."""
    return make_qk_workload(f"qwen_qk_{n_tokens}", n_tokens, 32, 4, 128, seed=seed)
