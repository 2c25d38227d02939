"""Python binding of librmsq (fused residual-add + RMSNorm + FP8 / NVFP4 quantisation).

Argument marshalling only: every step of the op runs in the library's CUDA
kernels.  torch is used for device memory and streams.  The names follow the C
ABI in ``include/rmsq.h``; if the built library is missing this module raises
instead of computing anything another way.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_lib", "librmsq.so")

# rmsq_status
OK, ERR_INVALID_ARG, ERR_ALIGNMENT, ERR_ALIAS, ERR_UNSUPPORTED_SHAPE, \
    ERR_UNSUPPORTED_DEVICE, ERR_NO_DEVICE, ERR_CUDA = range(8)

# rmsq_quant_mode
MODES = {
    "fp8_static": 0,
    "fp8_per_token": 1,
    "fp8_group128_row": 2,
    "fp8_group128_col": 3,
    "fp8_group64_row": 4,
    "fp8_group64_col": 5,
    "nvfp4": 6,
}
# Scale options (RMSQ_QUANT_E8M0, RMSQ_QUANT_TMA_ALIGNED, RMSQ_QUANT_UE8M0),
# appended to a mode name with "+": e.g. "fp8_group128_col+e8m0+tma",
# "fp8_per_token+ue8m0".
OPTIONS = {"e8m0": 0x10, "tma": 0x20, "ue8m0": 0x40}


def mode_code(mode: str) -> int:
    """The C quant_mode argument for a mode name with optional "+e8m0" / "+tma"."""
    base, *opts = mode.split("+")
    if base not in MODES or any(o not in OPTIONS for o in opts):
        raise ValueError(f"unknown quant mode {mode!r}")
    return MODES[base] | sum(OPTIONS[o] for o in opts)


def _variant(variant: str) -> int:
    if variant not in VARIANTS:
        raise ValueError(f"unknown variant {variant!r} (one of {', '.join(VARIANTS)})")
    return VARIANTS[variant]


# rmsq_dtype
DTYPES = {torch.bfloat16: 0, torch.float16: 1}
MAX_HIDDEN = 16384

VARIANTS = {"auto": 0, "direct": 1, "pipelined": 2}

EXPORTS = ("rmsq_fused_add_rmsnorm_quant", "rmsq_fused_add_rmsnorm_quant_ex",
           "rmsq_fused_add_rmsnorm_nvfp4_dynamic", "rmsq_nvfp4_dynamic_workspace_bytes",
           "rmsq_fused_add_rmsnorm_nvfp4_dynamic_noalloc", "rmsq_silu_mul_quant",
           "rmsq_fused_add_rmsnorm", "rmsq_quant", "rmsq_qk_norm_rope", "rmsq_qk_norm_rope_ex",
           "rmsq_allreduce_add_rmsnorm_quant",
           "rmsq_set_pipeline_config", "rmsq_set_programmatic_launch", "rmsq_take_fault_flags",
           "rmsq_query_sizes", "rmsq_query_launch", "rmsq_debug_convert", "rmsq_debug_activation", "rmsq_debug_bounded_wait",
           "rmsq_status_string", "rmsq_last_cuda_error", "rmsq_version")


class RmsqError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = status_string(status) if _lib is not None else str(status)
        if status == ERR_CUDA and _lib is not None:
            msg += f" (cudaError {_lib.rmsq_last_cuda_error()})"
        super().__init__(f"{where}: {msg} [status {status}]")


_lock = threading.Lock()
_lib = None


def load(path: str | None = None):
    """Load librmsq.so (built by ``residual_add_rmsnorm_rmsq_gb300._build.build()``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"librmsq.so not built ({p}); run residual_add_rmsnorm_rmsq_gb300._build.build()")
        L = ctypes.CDLL(p)
        vp, i64, f32, ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
        L.rmsq_fused_add_rmsnorm_quant.argtypes = [vp, vp, vp, f32, ci, vp, vp, vp, vp, i64, i64, ci, vp]
        L.rmsq_fused_add_rmsnorm_quant.restype = ci
        L.rmsq_fused_add_rmsnorm_quant_ex.argtypes = [vp, vp, vp, f32, ci, vp, vp, vp, vp, i64, i64, ci,
                                                      vp, ci]
        L.rmsq_fused_add_rmsnorm_quant_ex.restype = ci
        L.rmsq_fused_add_rmsnorm_nvfp4_dynamic.argtypes = [vp, vp, vp, f32, vp, vp, vp, vp, vp,
                                                           ctypes.c_size_t, i64, i64, ci, vp, ci]
        L.rmsq_fused_add_rmsnorm_nvfp4_dynamic.restype = ci
        L.rmsq_nvfp4_dynamic_workspace_bytes.argtypes = [i64]
        L.rmsq_nvfp4_dynamic_workspace_bytes.restype = ctypes.c_size_t
        L.rmsq_fused_add_rmsnorm.argtypes = [vp, vp, vp, f32, vp, vp, i64, i64, ci, vp]
        L.rmsq_fused_add_rmsnorm.restype = ci
        L.rmsq_qk_norm_rope.argtypes = [vp, vp, vp, i64, vp, vp, f32, i64, ci, ci, ci, ci, ci, vp]
        L.rmsq_qk_norm_rope.restype = ci
        L.rmsq_qk_norm_rope_ex.argtypes = [vp, vp, vp, i64, vp, vp, f32, i64, ci, ci, ci, ci, ci, vp, ci]
        L.rmsq_qk_norm_rope_ex.restype = ci
        L.rmsq_allreduce_add_rmsnorm_quant.argtypes = [ctypes.POINTER(vp), ci, vp, vp, f32, ci, vp, vp, vp, vp,
                                                       i64, i64, ci, vp]
        L.rmsq_allreduce_add_rmsnorm_quant.restype = ci
        L.rmsq_quant.argtypes = [vp, ci, vp, vp, vp, i64, i64, ci, vp]
        L.rmsq_quant.restype = ci
        L.rmsq_silu_mul_quant.argtypes = [vp, ci, vp, vp, vp, i64, i64, ci, vp]
        L.rmsq_silu_mul_quant.restype = ci
        L.rmsq_set_pipeline_config.argtypes = [ci, ci, ci, ci]
        L.rmsq_set_pipeline_config.restype = ci
        L.rmsq_set_programmatic_launch.argtypes = [ci]
        L.rmsq_set_programmatic_launch.restype = ci
        L.rmsq_take_fault_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
        L.rmsq_take_fault_flags.restype = ci
        L.rmsq_query_sizes.argtypes = [ci, i64, i64, ctypes.POINTER(ctypes.c_size_t),
                                       ctypes.POINTER(ctypes.c_size_t)]
        L.rmsq_query_sizes.restype = ci
        L.rmsq_query_launch.argtypes = [ci, i64, i64, ci, ci, ci, ctypes.POINTER(ctypes.c_int32)]
        L.rmsq_query_launch.restype = ci
        L.rmsq_debug_convert.argtypes = [ci, vp, vp, i64, vp]
        L.rmsq_debug_convert.restype = ci
        L.rmsq_debug_activation.argtypes = [ci, vp, vp, vp, i64, vp]
        L.rmsq_debug_activation.restype = ci
        L.rmsq_debug_bounded_wait.argtypes = [i64, ctypes.POINTER(ci)]
        L.rmsq_debug_bounded_wait.restype = ci
        L.rmsq_status_string.argtypes = [ci]
        L.rmsq_status_string.restype = ctypes.c_char_p
        L.rmsq_last_cuda_error.argtypes = []
        L.rmsq_last_cuda_error.restype = ci
        L.rmsq_version.argtypes = []
        L.rmsq_version.restype = ci
        _lib = L
        return L


def status_string(status: int) -> str:
    return load().rmsq_status_string(int(status)).decode()


def version() -> int:
    return load().rmsq_version()


def query_sizes(mode: str, n_tokens: int, hidden: int) -> tuple[int, int]:
    q, s = ctypes.c_size_t(), ctypes.c_size_t()
    st = load().rmsq_query_sizes(mode_code(mode), n_tokens, hidden, ctypes.byref(q), ctypes.byref(s))
    if st:
        raise RmsqError(st, "rmsq_query_sizes")
    return q.value, s.value


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def scales_like(mode: str, n_tokens: int, hidden: int, device) -> torch.Tensor | None:
    """An output tensor of the right shape and dtype for the scales of ``mode``
    (column-major with "+tma": [hidden/G, n_tokens rounded up to 16 bytes of
    scales]; uint8 with "+ue8m0")."""
    base, *opts = mode.split("+")
    if base == "fp8_static":
        return None
    if base == "nvfp4":
        return torch.empty(n_tokens, hidden // 16, dtype=torch.uint8, device=device)
    dt = torch.uint8 if "ue8m0" in opts else torch.float32
    if base == "fp8_per_token":
        return torch.empty(n_tokens, dtype=dt, device=device)
    G = 128 if "128" in base else 64
    per16 = 16 if "ue8m0" in opts else 4
    cols = (n_tokens + per16 - 1) // per16 * per16 if "tma" in opts else n_tokens
    shape = (hidden // G, cols) if base.endswith("_col") else (n_tokens, hidden // G)
    return torch.empty(shape, dtype=dt, device=device)


def fused_add_rmsnorm_quant(x: torch.Tensor, residual: torch.Tensor | None, weight: torch.Tensor,
                            eps: float, mode: str, scale_in: torch.Tensor | None = None, *,
                            out_q: torch.Tensor | None = None,
                            out_scales: torch.Tensor | None = None,
                            residual_out: torch.Tensor | None = None, stream=None,
                            variant: str = "auto"):
    """rmsq_fused_add_rmsnorm_quant on torch CUDA tensors.

    x, residual, residual_out: [n, H] bf16/fp16, contiguous; weight: [H];
    scale_in: fp32 device tensor with one element (FP8 static scale / NVFP4
    global scale).  Missing outputs are allocated.  Pass
    ``residual_out=residual`` for the in-place update.
    ``variant``: "auto", "direct" or "pipelined" (identical results).
    Returns (q, scales, residual_out).
    """
    vcode = _variant(variant)
    L = load()
    n, H = x.shape
    if x.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {x.dtype}")
    for t in (x, residual, weight, residual_out, out_q, out_scales, scale_in):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if out_q is None:
        out_q = torch.empty(n, H // 2 if mode == "nvfp4" else H, dtype=torch.uint8, device=x.device)
    if out_scales is None:
        out_scales = scales_like(mode, n, H, x.device)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(residual)
    st = L.rmsq_fused_add_rmsnorm_quant_ex(_p(x), _p(residual), _p(weight), ctypes.c_float(eps),
                                           mode_code(mode), _p(scale_in), _p(out_q), _p(out_scales),
                                           _p(residual_out), n, H, DTYPES[x.dtype], _stream(stream),
                                           vcode)
    if st:
        raise RmsqError(st, "rmsq_fused_add_rmsnorm_quant")
    return out_q, out_scales, residual_out


MAX_ALLREDUCE_RANKS = 8


def allreduce_add_rmsnorm_quant(partials, residual: torch.Tensor | None, weight: torch.Tensor, eps: float,
                                mode: str, scale_in: torch.Tensor | None = None, *,
                                out_q: torch.Tensor | None = None, out_scales: torch.Tensor | None = None,
                                residual_out: torch.Tensor | None = None, stream=None):
    """rmsq_allreduce_add_rmsnorm_quant: ``partials`` is a sequence of [n, H]
    tensors, one per rank (each readable by the current device), summed in
    rank order; then the fused op on the sum.  Returns (q, scales, residual_out)."""
    L = load()
    parts = list(partials)
    if not 1 <= len(parts) <= MAX_ALLREDUCE_RANKS:
        raise ValueError(f"1 to {MAX_ALLREDUCE_RANKS} partial tensors")
    x = parts[0]
    n, H = x.shape
    if x.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {x.dtype}")
    for t in parts:
        if t.shape != x.shape or t.dtype != x.dtype:
            raise ValueError("every partial must have the first one's shape and dtype")
    for t in parts + [residual, weight, residual_out, out_q, out_scales, scale_in]:
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if out_q is None:
        out_q = torch.empty(n, H // 2 if mode == "nvfp4" else H, dtype=torch.uint8, device=x.device)
    if out_scales is None:
        out_scales = scales_like(mode, n, H, x.device)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(residual)
    arr = (ctypes.c_void_p * len(parts))(*[t.data_ptr() for t in parts])
    st = L.rmsq_allreduce_add_rmsnorm_quant(arr, len(parts), _p(residual), _p(weight), ctypes.c_float(eps),
                                            mode_code(mode), _p(scale_in), _p(out_q), _p(out_scales),
                                            _p(residual_out), n, H, DTYPES[x.dtype], _stream(stream))
    if st:
        raise RmsqError(st, "rmsq_allreduce_add_rmsnorm_quant")
    return out_q, out_scales, residual_out


def row_slice(n_tokens: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [begin, end) of `rank` when `world` ranks split a batch for a
    two-shot all-reduce + norm (each rank reduces and normalises its slice,
    then the slices are gathered): contiguous, as equal as possible, the
    first n % world ranks one row longer."""
    if world < 1 or not 0 <= rank < world or n_tokens < 0:
        raise ValueError("bad world / rank / n_tokens")
    q, r = divmod(n_tokens, world)
    begin = rank * q + min(rank, r)
    return begin, begin + q + (1 if rank < r else 0)


def fused_add_rmsnorm(x: torch.Tensor, residual: torch.Tensor | None, weight: torch.Tensor, eps: float, *,
                      y_out: torch.Tensor | None = None, residual_out: torch.Tensor | None = None, stream=None):
    """rmsq_fused_add_rmsnorm: the norm alone, y in the activation type.
    Returns (y, residual_out)."""
    L = load()
    n, H = x.shape
    if x.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {x.dtype}")
    for t in (x, residual, weight, y_out, residual_out):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if y_out is None:
        y_out = torch.empty_like(x)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(residual)
    st = L.rmsq_fused_add_rmsnorm(_p(x), _p(residual), _p(weight), ctypes.c_float(eps), _p(y_out), _p(residual_out),
                                  n, H, DTYPES[x.dtype], _stream(stream))
    if st:
        raise RmsqError(st, "rmsq_fused_add_rmsnorm")
    return y_out, residual_out


def quant(y: torch.Tensor, mode: str, scale_in: torch.Tensor | None = None, *, out_q: torch.Tensor | None = None,
          out_scales: torch.Tensor | None = None, stream=None):
    """rmsq_quant: the quantisation of a [n, H] activation-type tensor.
    Returns (q, scales)."""
    L = load()
    n, H = y.shape
    if y.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {y.dtype}")
    for t in (y, out_q, out_scales, scale_in):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if out_q is None:
        out_q = torch.empty(n, H // 2 if mode == "nvfp4" else H, dtype=torch.uint8, device=y.device)
    if out_scales is None:
        out_scales = scales_like(mode, n, H, y.device)
    st = L.rmsq_quant(_p(y), mode_code(mode), _p(scale_in), _p(out_q), _p(out_scales), n, H, DTYPES[y.dtype],
                      _stream(stream))
    if st:
        raise RmsqError(st, "rmsq_quant")
    return out_q, out_scales


def qk_norm_rope(qkv: torch.Tensor, positions: torch.Tensor, cos_sin_cache: torch.Tensor, q_weight: torch.Tensor,
                 k_weight: torch.Tensor, eps: float, num_q_heads: int, num_kv_heads: int, head_dim: int,
                 is_neox: bool = True, stream=None, variant: str = "auto") -> torch.Tensor:
    """rmsq_qk_norm_rope_ex on torch CUDA tensors, in place on qkv (returned);
    variant "auto", "direct" or "pipelined" (bit-identical results)."""
    vcode = _variant(variant)
    L = load()
    if qkv.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {qkv.dtype}")
    for t in (qkv, positions, cos_sin_cache, q_weight, k_weight):
        if not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if positions.dtype != torch.int64 or cos_sin_cache.dtype != torch.float32:
        raise TypeError("positions must be int64 and cos_sin_cache float32")
    n = qkv.shape[0]
    st = L.rmsq_qk_norm_rope_ex(_p(qkv), _p(positions), _p(cos_sin_cache), cos_sin_cache.shape[0],
                                _p(q_weight), _p(k_weight), ctypes.c_float(eps), n, num_q_heads, num_kv_heads,
                                head_dim, 1 if is_neox else 0, DTYPES[qkv.dtype], _stream(stream),
                                vcode)
    if st:
        raise RmsqError(st, "rmsq_qk_norm_rope_ex")
    return qkv


def silu_mul_quant(gate_up: torch.Tensor, mode: str, scale_in: torch.Tensor | None = None, *,
                   out_q: torch.Tensor | None = None, out_scales: torch.Tensor | None = None, stream=None):
    """rmsq_silu_mul_quant on torch CUDA tensors: gate_up [n, 2d] (gate | up),
    scale_in a one-element fp32 device tensor (FP8 static scale / NVFP4 global
    scale).  Missing outputs are allocated.  Returns (q, scales)."""
    L = load()
    n, d2 = gate_up.shape
    if gate_up.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {gate_up.dtype}")
    if d2 % 2:
        raise ValueError("gate_up must have an even number of columns (gate | up)")
    d = d2 // 2
    for t in (gate_up, out_q, out_scales, scale_in):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    if out_q is None:
        out_q = torch.empty(n, d // 2 if mode == "nvfp4" else d, dtype=torch.uint8, device=gate_up.device)
    if out_scales is None:
        out_scales = scales_like(mode, n, d, gate_up.device)
    st = L.rmsq_silu_mul_quant(_p(gate_up), mode_code(mode), _p(scale_in), _p(out_q), _p(out_scales), n, d,
                               DTYPES[gate_up.dtype], _stream(stream))
    if st:
        raise RmsqError(st, "rmsq_silu_mul_quant")
    return out_q, out_scales


def nvfp4_dynamic_workspace_bytes(n_tokens: int) -> int:
    return load().rmsq_nvfp4_dynamic_workspace_bytes(n_tokens)


def fused_add_rmsnorm_nvfp4_dynamic(x: torch.Tensor, residual: torch.Tensor | None,
                                    weight: torch.Tensor, eps: float, *,
                                    out_q: torch.Tensor | None = None,
                                    out_scales: torch.Tensor | None = None,
                                    out_global_scale: torch.Tensor | None = None,
                                    residual_out: torch.Tensor | None = None,
                                    workspace: torch.Tensor | None = None, stream=None,
                                    variant: str = "auto"):
    """rmsq_fused_add_rmsnorm_nvfp4_dynamic on torch CUDA tensors: NVFP4 with
    gs = 2688 / amax(all y) computed on the device.  Missing outputs and the
    workspace are allocated.  Returns (q, block_scales, global_scale, residual_out)."""
    vcode = _variant(variant)
    L = load()
    n, H = x.shape
    if x.dtype not in DTYPES:
        raise TypeError(f"unsupported activation dtype {x.dtype}")
    for t in (x, residual, weight, residual_out, out_q, out_scales, out_global_scale, workspace):
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")
    dev = x.device
    if out_q is None:
        out_q = torch.empty(n, H // 2, dtype=torch.uint8, device=dev)
    if out_scales is None:
        out_scales = torch.empty(n, H // 16, dtype=torch.uint8, device=dev)
    if out_global_scale is None:
        out_global_scale = torch.empty(1, dtype=torch.float32, device=dev)
    if residual is not None and residual_out is None:
        residual_out = torch.empty_like(residual)
    ws_bytes = nvfp4_dynamic_workspace_bytes(n)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 16), dtype=torch.uint8, device=dev)
    st = L.rmsq_fused_add_rmsnorm_nvfp4_dynamic(
        _p(x), _p(residual), _p(weight), ctypes.c_float(eps), _p(out_q), _p(out_scales),
        _p(out_global_scale), _p(residual_out), _p(workspace),
        workspace.numel() * workspace.element_size(), n, H, DTYPES[x.dtype], _stream(stream),
        vcode)
    if st:
        raise RmsqError(st, "rmsq_fused_add_rmsnorm_nvfp4_dynamic")
    return out_q, out_scales, out_global_scale, residual_out


def query_launch(mode: str, n_tokens: int, hidden: int, residual: bool = True, dtype=torch.bfloat16,
                 variant: str = "auto") -> dict:
    """rmsq_query_launch: the launch the fused op would make on the current
    device for this mode and shape (kernel variant, chunks per thread, ring
    stages, CTAs, threads per CTA); nothing is launched."""
    out = (ctypes.c_int32 * 5)()
    st = load().rmsq_query_launch(mode_code(mode), n_tokens, hidden, 1 if residual else 0, DTYPES[dtype],
                                  _variant(variant), out)
    if st:
        raise RmsqError(st, "rmsq_query_launch")
    return {"pipelined": bool(out[0]), "chunks_per_thread": out[1], "stages": out[2], "ctas": out[3],
            "threads": out[4]}


def set_pipeline_config(chunks_per_thread: int = 0, stages: int = 0, ctas_per_sm: int = 0,
                        rows_per_iter: int = 0) -> None:
    """Tune the pipelined variant's launch shape (0 = automatic); results are unchanged."""
    st = load().rmsq_set_pipeline_config(chunks_per_thread, stages, ctas_per_sm, rows_per_iter)
    if st:
        raise RmsqError(st, "rmsq_set_pipeline_config")


def set_programmatic_launch(enable: bool) -> None:
    """Launch with programmatic dependent launch (default) or plain stream order."""
    st = load().rmsq_set_programmatic_launch(1 if enable else 0)
    if st:
        raise RmsqError(st, "rmsq_set_programmatic_launch")


def take_fault_flags() -> int:
    """Read and clear the pipelined kernels' give-up flag (0 = none)."""
    f = ctypes.c_uint32()
    st = load().rmsq_take_fault_flags(ctypes.byref(f))
    if st:
        raise RmsqError(st, "rmsq_take_fault_flags")
    return f.value


def debug_activation(kind: str, values: torch.Tensor, up: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """The library's e^x ("exp"; "exp_mid": the steps used for |x| <= 87),
    silu ("silu") or silu(g) * u ("silu_mul") on fp32 CUDA tensors, elementwise."""
    L = load()
    v = values.contiguous().float()
    u = None if up is None else up.contiguous().float()
    out = torch.empty(v.shape, dtype=torch.float32, device=v.device)
    st = L.rmsq_debug_activation({"exp": 0, "silu": 1, "silu_mul": 2, "exp_mid": 3}[kind], _p(v), _p(u), _p(out), v.numel(),
                                 _stream(stream))
    if st:
        raise RmsqError(st, "rmsq_debug_activation")
    return out


def debug_bounded_wait(limit_ns: int) -> int:
    """Run the bounded-wait check (rmsq_debug_bounded_wait); returns gave_up."""
    out = ctypes.c_int(-1)
    st = load().rmsq_debug_bounded_wait(int(limit_ns), ctypes.byref(out))
    if st:
        raise RmsqError(st, "rmsq_debug_bounded_wait")
    return out.value


def debug_convert(kind: str, values: torch.Tensor, stream=None) -> torch.Tensor:
    """The library's E4M3 ("e4m3") or E2M1 ("e2m1", low nibble) conversion of a
    fp32 CUDA tensor."""
    L = load()
    v = values.contiguous().float()
    out = torch.empty(v.shape, dtype=torch.uint8, device=v.device)
    st = L.rmsq_debug_convert({"e4m3": 0, "e2m1": 1}[kind], _p(v), _p(out), v.numel(), _stream(stream))
    if st:
        raise RmsqError(st, "rmsq_debug_convert")
    return out
