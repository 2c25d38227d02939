"""CPU oracle for the fused residual-add + RMSNorm + quantisation op (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: imported by the tests, by the smoke check and by the
benchmark's CPU-baseline / reference leg, never by the library.  The C source
(``rmsq_oracle.c``) holds the definition and the passages it follows; it shares
no code with the CUDA path.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "rmsq_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_rmsq.so")

# The oracle's own names for the quantisation modes and activation types.
MODES = {
    "fp8_static": 0,
    "fp8_per_token": 1,
    "fp8_group128_row": 2,
    "fp8_group128_col": 3,
    "fp8_group64_row": 4,
    "fp8_group64_col": 5,
    "nvfp4": 6,
}
DTYPES = {"bf16": 0, "fp16": 1}
# Scale options, appended to a mode name with "+": "e8m0" (dynamic scales
# rounded up to a power of two), "ue8m0" (those scales stored as one UE8M0
# byte each) and "tma" (column-major scales with the stride padded to 16
# bytes: a multiple of 4 fp32 scales or of 16 bytes).
OPTIONS = {"e8m0": 0x10, "tma": 0x20, "ue8m0": 0x40}


def mode_code(mode: str) -> int:
    """The oracle's integer for a mode name with optional "+e8m0" / "+tma"."""
    base, *opts = mode.split("+")
    return MODES[base] | sum(OPTIONS[o] for o in opts)


def base_mode(mode: str) -> str:
    return mode.split("+")[0]
GROUP = {"fp8_group128_row": 128, "fp8_group128_col": 128,
         "fp8_group64_row": 64, "fp8_group64_col": 64}

_lock = threading.Lock()
_lib = None


def compile_oracle(force: bool = False) -> str:
    """gcc -O2 -ffp-contract=off, no fast-math: binary32 RNE, no contraction."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", "-pthread", _SRC, "-o", tmp, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    """The oracle library; ORACLE_LIB=<path> loads another build of the same
    source instead (used by the planted-mistake tests)."""
    global _lib
    with _lock:
        if _lib is None:
            path = os.environ.get("ORACLE_LIB") or compile_oracle()
            _lib = _configure(ctypes.CDLL(path))
    return _lib


class use_library:
    """Context manager: route every oracle call to another build of the C
    source (the tests use it to plant mistakes and check the pins catch them)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        lib()
        self.saved = _lib
        _lib = _configure(ctypes.CDLL(self.path))
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self.saved
        return False


def _configure(L):
    """Declare the C signatures on a loaded oracle library."""
    f32, u8, u16, i64, vp = (ctypes.c_float, ctypes.c_uint8, ctypes.c_uint16,
                             ctypes.c_int64, ctypes.c_void_p)
    L.oracle_bf16_to_float.argtypes, L.oracle_bf16_to_float.restype = [u16], f32
    L.oracle_fp16_to_float.argtypes, L.oracle_fp16_to_float.restype = [u16], f32
    L.oracle_float_to_bf16.argtypes, L.oracle_float_to_bf16.restype = [f32], u16
    L.oracle_float_to_fp16.argtypes, L.oracle_float_to_fp16.restype = [f32], u16
    L.oracle_e4m3_encode.argtypes, L.oracle_e4m3_encode.restype = [f32], u8
    L.oracle_e4m3_decode.argtypes, L.oracle_e4m3_decode.restype = [u8], f32
    L.oracle_e2m1_encode.argtypes, L.oracle_e2m1_encode.restype = [f32], u8
    L.oracle_e2m1_decode.argtypes, L.oracle_e2m1_decode.restype = [u8], f32
    L.oracle_tree_sum.argtypes, L.oracle_tree_sum.restype = [vp, i64], f32
    for name in ("oracle_e4m3_encode_array", "oracle_e2m1_encode_array",
                 "oracle_float_to_bf16_array", "oracle_float_to_fp16_array"):
        getattr(L, name).argtypes = [vp, vp, i64]
        getattr(L, name).restype = None
    L.oracle_fused_add_rmsnorm_quant.argtypes = [
        vp, vp, vp, f32, ctypes.c_int, f32, vp, vp, vp, vp, i64, i64, ctypes.c_int,
        ctypes.c_int]
    L.oracle_fused_add_rmsnorm_quant.restype = ctypes.c_int
    L.oracle_fused_add_rmsnorm_nvfp4_dynamic.argtypes = [
        vp, vp, vp, f32, vp, vp, vp, vp, i64, i64, ctypes.c_int, ctypes.c_int]
    L.oracle_fused_add_rmsnorm_nvfp4_dynamic.restype = ctypes.c_int
    L.oracle_silu_mul_quant.argtypes = [vp, ctypes.c_int, f32, vp, vp, vp, i64, i64, ctypes.c_int,
                                        ctypes.c_int]
    L.oracle_silu_mul_quant.restype = ctypes.c_int
    L.oracle_add_rmsnorm.argtypes = [vp, vp, vp, f32, vp, vp, i64, i64, ctypes.c_int, ctypes.c_int]
    L.oracle_add_rmsnorm.restype = ctypes.c_int
    L.oracle_quant.argtypes = [vp, ctypes.c_int, f32, vp, vp, i64, i64, ctypes.c_int, ctypes.c_int]
    L.oracle_quant.restype = ctypes.c_int
    L.oracle_qk_norm_rope.argtypes = [vp, vp, vp, i64, vp, vp, f32, i64, ctypes.c_int, ctypes.c_int,
                                      ctypes.c_int, ctypes.c_int, ctypes.c_int]
    L.oracle_qk_norm_rope.restype = ctypes.c_int
    L.oracle_silu.argtypes, L.oracle_silu.restype = [f32], f32
    L.oracle_silu_array.argtypes = [vp, vp, i64]
    L.oracle_silu_array.restype = None
    L.oracle_allreduce_add_rmsnorm_quant.argtypes = [vp, ctypes.c_int, vp, vp, f32, ctypes.c_int, f32, vp, vp, vp,
                                                     vp, i64, i64, ctypes.c_int, ctypes.c_int]
    L.oracle_allreduce_add_rmsnorm_quant.restype = ctypes.c_int
    L.oracle_quant_f32.argtypes = [vp, ctypes.c_int, f32, vp, vp, i64, i64, ctypes.c_int]
    L.oracle_quant_f32.restype = ctypes.c_int
    return L


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def e4m3_encode(v) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e2m1_encode(v) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e2m1_encode_array(_ptr(v), _ptr(out), v.size)
    return out


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e4m3_decode(int(c)) for c in np.ravel(codes)],
                    np.float32).reshape(np.shape(codes))


def e2m1_decode(codes) -> np.ndarray:
    L = lib()
    return np.array([L.oracle_e2m1_decode(int(c)) for c in np.ravel(codes)],
                    np.float32).reshape(np.shape(codes))


def float_to_act(v, dtype: str) -> np.ndarray:
    v = _f32(v)
    out = np.empty(v.shape, np.uint16)
    fn = lib().oracle_float_to_bf16_array if dtype == "bf16" else lib().oracle_float_to_fp16_array
    fn(_ptr(v), _ptr(out), v.size)
    return out


def act_to_float(bits, dtype: str) -> np.ndarray:
    L = lib()
    fn = L.oracle_bf16_to_float if dtype == "bf16" else L.oracle_fp16_to_float
    return np.array([fn(int(b)) for b in np.ravel(bits)], np.float32).reshape(np.shape(bits))


def tree_sum(v) -> float:
    v = _f32(v)
    return float(lib().oracle_tree_sum(_ptr(v), v.size))


def scale_shape(mode: str, n: int, H: int):
    """Shape and dtype of the scale output of ``mode`` for an [n, H] input
    (column-major with "+tma": [H/G, n rounded up to 4], or to 16 with
    "+ue8m0"; one uint8 per scale with "+ue8m0")."""
    base = base_mode(mode)
    if base == "fp8_static":
        return None
    if base == "nvfp4":
        return (n, H // 16), np.uint8
    opts = mode.split("+")[1:]
    dt = np.uint8 if "ue8m0" in opts else np.float32
    if base == "fp8_per_token":
        return (n,), dt
    G = GROUP[base]
    if base.endswith("_col"):
        per16 = 16 if "ue8m0" in opts else 4
        return (H // G, (n + per16 - 1) // per16 * per16 if "tma" in opts else n), dt
    return (n, H // G), dt


def run(x, residual, weight, *, eps: float, mode: str, scale_in: float = 0.0,
        dtype: str = "bf16", want_y: bool = False, nthreads: int = 1) -> dict:
    """Run the oracle on host bit patterns (uint16 [n, H], [n, H] or None, [H]).

    Returns a dict with ``q`` (uint8 [n, H] for FP8, [n, H/2] for NVFP4),
    ``scales`` (None for FP8 static), ``residual_out`` (None without a
    residual) and, when ``want_y``, the fp32 ``y`` [n, H].
    """
    x = np.ascontiguousarray(x, np.uint16)
    n, H = x.shape
    weight = np.ascontiguousarray(weight, np.uint16)
    assert weight.shape == (H,)
    res = None if residual is None else np.ascontiguousarray(residual, np.uint16)
    q = np.zeros((n, H // 2) if mode == "nvfp4" else (n, H), np.uint8)
    ss = scale_shape(mode, n, H)
    scales = None if ss is None else np.zeros(ss[0], ss[1])
    res_out = None if res is None else np.zeros((n, H), np.uint16)
    y = np.zeros((n, H), np.float32) if want_y else None
    rc = lib().oracle_fused_add_rmsnorm_quant(
        _ptr(x), _ptr(res), _ptr(weight), ctypes.c_float(eps), mode_code(mode),
        ctypes.c_float(scale_in), _ptr(q), _ptr(scales), _ptr(res_out), _ptr(y),
        n, H, DTYPES[dtype], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"q": q, "scales": scales, "residual_out": res_out, "y": y}


def run_allreduce(partials, residual, weight, *, eps: float, mode: str, scale_in: float = 0.0,
                  dtype: str = "bf16", want_y: bool = False, nthreads: int = 1) -> dict:
    """All-reduce + the fused op (reading R22): ``partials`` uint16 [R, n, H]
    (one [n, H] tensor per rank); outputs as for ``run``."""
    p = np.ascontiguousarray(partials, np.uint16)
    R, n, H = p.shape
    weight = np.ascontiguousarray(weight, np.uint16)
    res = None if residual is None else np.ascontiguousarray(residual, np.uint16)
    q = np.zeros((n, H // 2) if base_mode(mode) == "nvfp4" else (n, H), np.uint8)
    ss = scale_shape(mode, n, H)
    scales = None if ss is None else np.zeros(ss[0], ss[1])
    res_out = None if res is None else np.zeros((n, H), np.uint16)
    y = np.zeros((n, H), np.float32) if want_y else None
    rc = lib().oracle_allreduce_add_rmsnorm_quant(
        _ptr(p), R, _ptr(res), _ptr(weight), ctypes.c_float(eps), mode_code(mode), ctypes.c_float(scale_in),
        _ptr(q), _ptr(scales), _ptr(res_out), _ptr(y), n, H, DTYPES[dtype], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"q": q, "scales": scales, "residual_out": res_out, "y": y}


def run_nvfp4_dynamic(x, residual, weight, *, eps: float, dtype: str = "bf16",
                      nthreads: int = 1) -> dict:
    """NVFP4 with gs = 2688 / amax(all y) computed inside the oracle (1 when
    amax is 0).  Returns q, scales (block scales), residual_out and gs."""
    x = np.ascontiguousarray(x, np.uint16)
    n, H = x.shape
    weight = np.ascontiguousarray(weight, np.uint16)
    res = None if residual is None else np.ascontiguousarray(residual, np.uint16)
    q = np.zeros((n, H // 2), np.uint8)
    sc = np.zeros((n, H // 16), np.uint8)
    ro = None if res is None else np.zeros((n, H), np.uint16)
    gs = np.zeros(1, np.float32)
    rc = lib().oracle_fused_add_rmsnorm_nvfp4_dynamic(
        _ptr(x), _ptr(res), _ptr(weight), ctypes.c_float(eps), _ptr(q), _ptr(sc), _ptr(gs),
        _ptr(ro), n, H, DTYPES[dtype], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"q": q, "scales": sc, "residual_out": ro, "global_scale": gs}


def silu(v) -> np.ndarray:
    """silu(g) = g / (1 + e^-g) elementwise: evaluated in binary64, rounded once
    to binary32 (reading R15)."""
    v = _f32(v)
    out = np.empty(v.shape, np.float32)
    lib().oracle_silu_array(_ptr(v), _ptr(out), v.size)
    return out


def run_silu_mul(gate_up, *, mode: str, scale_in: float = 0.0, dtype: str = "bf16",
                 want_y: bool = False, nthreads: int = 1) -> dict:
    """SiLU+Mul + quantisation on host bit patterns: gate_up uint16 [n, 2d]
    (gate in the first d columns, up in the next d).  Returns ``q``,
    ``scales`` and, when ``want_y``, the fp32 activation ``y`` [n, d]."""
    gu = np.ascontiguousarray(gate_up, np.uint16)
    n, d2 = gu.shape
    assert d2 % 2 == 0
    d = d2 // 2
    q = np.zeros((n, d // 2) if mode == "nvfp4" else (n, d), np.uint8)
    ss = scale_shape(mode, n, d)
    scales = None if ss is None else np.zeros(ss[0], ss[1])
    y = np.zeros((n, d), np.float32) if want_y else None
    rc = lib().oracle_silu_mul_quant(_ptr(gu), mode_code(mode), ctypes.c_float(scale_in), _ptr(q), _ptr(scales),
                                     _ptr(y), n, d, DTYPES[dtype], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"q": q, "scales": scales, "residual_out": None, "y": y}


def run_quant_f32(y, *, mode: str, scale_in: float = 0.0, nthreads: int = 1) -> dict:
    """The quantisation step alone on given fp32 rows y [n, d] (any producer's
    activations): ``q`` and ``scales`` laid out as for the fused op."""
    y = np.ascontiguousarray(y, np.float32)
    n, d = y.shape
    q = np.zeros((n, d // 2) if mode == "nvfp4" else (n, d), np.uint8)
    ss = scale_shape(mode, n, d)
    scales = None if ss is None else np.zeros(ss[0], ss[1])
    rc = lib().oracle_quant_f32(_ptr(y), mode_code(mode), ctypes.c_float(scale_in), _ptr(q), _ptr(scales), n, d,
                                int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"q": q, "scales": scales, "residual_out": None}


def run_silu_mul_workload(wl, mode: str, *, scale_in: float | None = None, want_y: bool = False,
                          nthreads: int = 1) -> dict:
    """Run a SiLU+Mul workload (``rmsq_inputs.ActWorkload``).  For NVFP4
    without an explicit scale_in, gs = 2688 / amax(all activations) from a
    first pass, as for the norm op."""
    if mode == "fp8_static" and scale_in is None:
        scale_in = wl.static_scale
    if mode == "nvfp4" and scale_in is None:
        pre = run_silu_mul(wl.gate_up, mode="fp8_per_token", dtype=wl.dtype, want_y=True, nthreads=nthreads)
        scale_in = nvfp4_global_scale(float(np.max(np.abs(pre["y"]))))
    r = run_silu_mul(wl.gate_up, mode=mode, scale_in=scale_in or 0.0, dtype=wl.dtype, want_y=want_y,
                     nthreads=nthreads)
    r["scale_in"] = scale_in
    return r


def run_add_rmsnorm(x, residual, weight, *, eps: float, dtype: str = "bf16", nthreads: int = 1) -> dict:
    """First op of the unfused sequence: ``y_t`` (y rounded to the activation
    type, uint16 bit patterns [n, H]) and ``residual_out``."""
    x = np.ascontiguousarray(x, np.uint16)
    n, H = x.shape
    weight = np.ascontiguousarray(weight, np.uint16)
    res = None if residual is None else np.ascontiguousarray(residual, np.uint16)
    y_t = np.zeros((n, H), np.uint16)
    ro = None if res is None else np.zeros((n, H), np.uint16)
    rc = lib().oracle_add_rmsnorm(_ptr(x), _ptr(res), _ptr(weight), ctypes.c_float(eps), _ptr(y_t), _ptr(ro),
                                  n, H, DTYPES[dtype], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"y_t": y_t, "residual_out": ro}


def run_quant(y_t, *, mode: str, scale_in: float = 0.0, dtype: str = "bf16", nthreads: int = 1) -> dict:
    """Second op of the unfused sequence: the quantisation of a T tensor."""
    y_t = np.ascontiguousarray(y_t, np.uint16)
    n, H = y_t.shape
    q = np.zeros((n, H // 2) if base_mode(mode) == "nvfp4" else (n, H), np.uint8)
    ss = scale_shape(mode, n, H)
    scales = None if ss is None else np.zeros(ss[0], ss[1])
    rc = lib().oracle_quant(_ptr(y_t), mode_code(mode), ctypes.c_float(scale_in), _ptr(q), _ptr(scales), n, H,
                            DTYPES[dtype], int(nthreads))
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return {"q": q, "scales": scales, "residual_out": None}


def run_qk_norm_rope(wl) -> np.ndarray:
    """QK-norm + RoPE on a ``rmsq_inputs.QKWorkload``; returns the updated
    qkv bit patterns (uint16 [n, (nq + 2 nkv) D])."""
    qkv = np.ascontiguousarray(wl.qkv, np.uint16).copy()
    pos = np.ascontiguousarray(wl.positions, np.int64)
    cs = np.ascontiguousarray(wl.cos_sin, np.float32)
    rc = lib().oracle_qk_norm_rope(_ptr(qkv), _ptr(pos), _ptr(cs), cs.shape[0], _ptr(wl.q_weight),
                                   _ptr(wl.k_weight), ctypes.c_float(wl.eps), wl.n_tokens, wl.nq, wl.nkv,
                                   wl.head_dim, 1 if wl.neox else 0, DTYPES[wl.dtype])
    if rc != 0:
        raise RuntimeError(f"oracle failed with code {rc}")
    return qkv


def nvfp4_global_scale(y_amax: float) -> float:
    """gs = 448 * 6 / amax(all y), as the NVFP4 workload defines it (fp32 division)."""
    return float(np.float32(2688.0) / np.float32(y_amax))


def run_workload(wl, mode: str, *, scale_in: float | None = None, want_y: bool = False,
                 nthreads: int = 1) -> dict:
    """Run a ``rmsq_inputs.Workload``.  For NVFP4 without an explicit scale_in,
    a first pass computes y and sets gs = 2688 / amax(all y)."""
    if mode == "fp8_static" and scale_in is None:
        scale_in = wl.static_scale
    out = None
    if mode == "nvfp4" and scale_in is None:
        pre = run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode="fp8_per_token",
                  dtype=wl.dtype, want_y=True, nthreads=nthreads)
        scale_in = nvfp4_global_scale(float(np.max(np.abs(pre["y"]))))
        if want_y:
            out = pre["y"]
    r = run(wl.x, wl.residual, wl.weight, eps=wl.eps, mode=mode, scale_in=scale_in or 0.0,
            dtype=wl.dtype, want_y=want_y and out is None, nthreads=nthreads)
    if out is not None:
        r["y"] = out
    r["scale_in"] = scale_in
    return r
