"""Host-side checks of the C ABI (no GPU needed, no kernel runs).

The library must load, export every entry point include/rmsq.h declares, and
reject bad arguments with the documented status before touching a device.
Pointers here are fake addresses: validation never dereferences them.
"""
import ctypes
import os
import re

import pytest
import torch

import residual_add_rmsnorm_rmsq_gb300 as rq

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "rmsq.h")


@pytest.fixture(scope="module")
def L():
    from residual_add_rmsnorm_rmsq_gb300 import _build
    _build.build()
    return rq.load()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:int|size_t|const char \*)\s*(rmsq_\w+)\s*\(", src, flags=re.M)))


def test_every_declared_symbol_is_exported(L):
    names = _declared()
    assert set(names) == set(rq.EXPORTS), names
    for n in names:
        assert hasattr(L, n), n


def test_version_and_status_strings(L):
    assert rq.version() == 10000
    for s in range(8):
        assert rq.status_string(s)
    assert rq.status_string(99) == "unknown status"


def test_query_sizes(L):
    assert rq.query_sizes("fp8_static", 4, 64) == (256, 0)
    assert rq.query_sizes("fp8_per_token", 4, 64) == (256, 16)
    assert rq.query_sizes("fp8_group128_row", 3, 256) == (768, 24)
    assert rq.query_sizes("fp8_group64_col", 3, 256) == (768, 48)
    assert rq.query_sizes("nvfp4", 5, 2048) == (5 * 1024, 5 * 128)
    with pytest.raises(rq.RmsqError):
        rq.query_sizes("nvfp4", 5, 40)
    # scale options: E8M0 keeps the sizes, TMA alignment pads the column stride to 4
    assert rq.query_sizes("fp8_group64_col+e8m0", 3, 256) == (768, 48)
    assert rq.query_sizes("fp8_group64_col+tma", 3, 256) == (768, 4 * 4 * 4)
    assert rq.query_sizes("fp8_group128_col+e8m0+tma", 9, 256) == (9 * 256, 2 * 12 * 4)
    # UE8M0 bytes: one byte per scale; with TMA alignment the stride pads to 16
    assert rq.query_sizes("fp8_per_token+ue8m0", 4, 64) == (256, 4)
    assert rq.query_sizes("fp8_group64_row+ue8m0", 3, 256) == (768, 12)
    assert rq.query_sizes("fp8_group128_col+ue8m0+tma", 9, 256) == (9 * 256, 2 * 16)
    assert rq.query_sizes("fp8_group128_col+ue8m0+tma", 17, 256) == (17 * 256, 2 * 32)
    for bad in ("fp8_static+ue8m0", "nvfp4+ue8m0"):
        with pytest.raises(rq.RmsqError) as ei:
            rq.query_sizes(bad, 4, 256)
        assert ei.value.status == rq.ERR_INVALID_ARG


A, B, C, D, E, F = (0x10000000 * k for k in range(1, 7))   # far-apart fake addresses


def call(L, x=A, res=B, w=C, eps=1e-6, mode=1, s_in=None, q=D, sc=E, ro=F, n=4, H=64, dt=0):
    vp = ctypes.c_void_p
    return L.rmsq_fused_add_rmsnorm_quant(vp(x) if x else None, vp(res) if res else None,
                                          vp(w) if w else None, ctypes.c_float(eps), mode,
                                          vp(s_in) if s_in else None, vp(q) if q else None,
                                          vp(sc) if sc else None, vp(ro) if ro else None,
                                          n, H, dt, None)


def test_byte_scales_need_no_word_alignment(L):
    """fp32 scales must start on 4 bytes; UE8M0 bytes on any address (the
    call then fails only on the missing device, after every argument check)."""
    assert call(L, mode=1, sc=E + 2) == rq.ERR_ALIGNMENT
    assert call(L, mode=1 | 0x40, sc=E + 2) in (rq.ERR_NO_DEVICE, rq.ERR_UNSUPPORTED_DEVICE)


def test_argument_errors(L):
    assert call(L, dt=2) == rq.ERR_INVALID_ARG
    assert call(L, mode=7) == rq.ERR_INVALID_ARG
    assert call(L, mode=-1) == rq.ERR_INVALID_ARG
    assert call(L, n=-1) == rq.ERR_INVALID_ARG
    assert call(L, H=0) == rq.ERR_INVALID_ARG
    assert call(L, eps=-1.0) == rq.ERR_INVALID_ARG
    assert call(L, eps=float("nan")) == rq.ERR_INVALID_ARG
    assert call(L, eps=float("inf")) == rq.ERR_INVALID_ARG
    assert call(L, x=0) == rq.ERR_INVALID_ARG
    assert call(L, w=0) == rq.ERR_INVALID_ARG
    assert call(L, q=0) == rq.ERR_INVALID_ARG
    assert call(L, ro=0) == rq.ERR_INVALID_ARG           # residual without residual_out
    assert call(L, res=0) == rq.ERR_INVALID_ARG          # residual_out without residual
    assert call(L, sc=0) == rq.ERR_INVALID_ARG           # dynamic mode needs out_scales
    assert call(L, mode=0) == rq.ERR_INVALID_ARG         # static needs scale_in
    assert call(L, mode=6, H=64) == rq.ERR_INVALID_ARG   # NVFP4 needs scale_in
    # scale options only where they apply, no unknown bits
    assert call(L, mode=0x10 | 0, s_in=A + 0x100) == rq.ERR_INVALID_ARG   # E8M0 with a static scale
    assert call(L, mode=0x10 | 6, s_in=A + 0x100) == rq.ERR_INVALID_ARG   # E8M0 with NVFP4
    assert call(L, mode=0x20 | 2) == rq.ERR_INVALID_ARG                   # TMA with row-major scales
    assert call(L, mode=0x20 | 1) == rq.ERR_INVALID_ARG                   # TMA with per-token
    assert call(L, mode=0x80 | 1) == rq.ERR_INVALID_ARG                   # unknown bit
    assert call(L, mode=0x40 | 0, s_in=A + 0x100) == rq.ERR_INVALID_ARG   # UE8M0 with a static scale
    assert call(L, mode=0x10 | 1) == rq.ERR_NO_DEVICE                     # valid: reaches the device check
    assert call(L, mode=0x30 | 3, H=128) == rq.ERR_NO_DEVICE


def test_shape_errors(L):
    assert call(L, H=60) == rq.ERR_UNSUPPORTED_SHAPE
    assert call(L, H=16392) == rq.ERR_UNSUPPORTED_SHAPE
    assert call(L, mode=2, H=64) == rq.ERR_UNSUPPORTED_SHAPE
    assert call(L, mode=4, H=96) == rq.ERR_UNSUPPORTED_SHAPE
    assert call(L, mode=6, H=24, s_in=0x7000000) == rq.ERR_UNSUPPORTED_SHAPE
    assert call(L, n=2 ** 31) == rq.ERR_UNSUPPORTED_SHAPE


def test_empty_input_is_ok_without_pointers(L):
    assert call(L, n=0, x=0, res=0, w=0, q=0, sc=0, ro=0) == rq.OK


def test_alignment_errors(L):
    assert call(L, x=A + 8) == rq.ERR_ALIGNMENT
    assert call(L, res=B + 2) == rq.ERR_ALIGNMENT
    assert call(L, w=C + 4) == rq.ERR_ALIGNMENT
    assert call(L, q=D + 8) == rq.ERR_ALIGNMENT
    assert call(L, ro=F + 8) == rq.ERR_ALIGNMENT
    assert call(L, sc=E + 2) == rq.ERR_ALIGNMENT
    assert call(L, mode=0, s_in=E + 2, sc=0) == rq.ERR_ALIGNMENT


def test_alias_errors(L):
    act = 4 * 64 * 2
    assert call(L, ro=B + 16) == rq.ERR_ALIAS               # partial overlap with residual
    assert call(L, res=A + 16, ro=F) == rq.ERR_ALIAS        # x and residual partially overlap
    assert call(L, q=A + act - 16) == rq.ERR_ALIAS          # codes over x
    assert call(L, sc=D + 128) == rq.ERR_ALIAS              # scales over codes
    assert call(L, ro=C) == rq.ERR_ALIAS                    # residual_out over weight
    assert call(L, q=F + 64) == rq.ERR_ALIAS                # codes over residual_out


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_call_without_device_reports_no_device(L):
    assert call(L) == rq.ERR_NO_DEVICE
    assert call(L, ro=B) == rq.ERR_NO_DEVICE                 # in place: allowed
    assert call(L, ro=A) == rq.ERR_NO_DEVICE                 # over x: allowed
    assert call(L, mode=0, s_in=0x7000000, sc=0) == rq.ERR_NO_DEVICE
    vp = ctypes.c_void_p
    assert L.rmsq_debug_convert(0, vp(A), vp(B), 16, None) == rq.ERR_NO_DEVICE
    assert L.rmsq_debug_convert(2, vp(A), vp(B), 16, None) == rq.ERR_INVALID_ARG


def test_nvfp4_dynamic_argument_errors(L):
    vp = ctypes.c_void_p
    ws = rq.nvfp4_dynamic_workspace_bytes(4)
    # 256 + 8 n rounded up to 256: a header, an inverse RMS and a partial maximum per row
    assert ws == 512 and rq.nvfp4_dynamic_workspace_bytes(32) == 512
    assert rq.nvfp4_dynamic_workspace_bytes(33) == 768 and rq.nvfp4_dynamic_workspace_bytes(0) == 256

    def dyn(x=A, res=B, w=C, q=D, sc=E, gs=0x70000000, ro=F, wsp=0x78000000, wsb=ws, n=4, H=64, dt=0, v=0):
        return L.rmsq_fused_add_rmsnorm_nvfp4_dynamic(
            vp(x) if x else None, vp(res) if res else None, vp(w) if w else None, ctypes.c_float(1e-6),
            vp(q) if q else None, vp(sc) if sc else None, vp(gs) if gs else None, vp(ro) if ro else None,
            vp(wsp) if wsp else None, wsb, n, H, dt, None, v)

    assert dyn(H=40) == rq.ERR_UNSUPPORTED_SHAPE
    assert dyn(wsp=0) == rq.ERR_INVALID_ARG
    assert dyn(wsb=ws - 1) == rq.ERR_INVALID_ARG
    assert dyn(gs=0) == rq.ERR_INVALID_ARG
    assert dyn(v=3) == rq.ERR_INVALID_ARG
    assert dyn(wsp=0x78000000 + 8) == rq.ERR_ALIGNMENT
    assert dyn(gs=0x70000000 + 2) == rq.ERR_ALIGNMENT
    assert dyn(wsp=D) == rq.ERR_ALIAS                      # workspace over the codes
    assert dyn(gs=E + 4) == rq.ERR_ALIAS                    # global scale inside block scales
    assert dyn(n=0, x=0, res=0, w=0, q=0, sc=0, gs=0, ro=0, wsp=0) == rq.OK
    if not torch.cuda.is_available():
        assert dyn() == rq.ERR_NO_DEVICE


def test_silu_mul_quant_argument_errors(L):
    vp = ctypes.c_void_p
    GU, Q, SC, SI = 0x50000000, 0x51000000, 0x52000000, 0x53000000

    def act(gu=GU, mode=1, si=0, q=Q, sc=SC, n=4, d=64, dt=0):
        return L.rmsq_silu_mul_quant(vp(gu) if gu else None, mode, vp(si) if si else None, vp(q) if q else None,
                                     vp(sc) if sc else None, n, d, dt, None)

    assert act(dt=2) == rq.ERR_INVALID_ARG
    assert act(mode=7) == rq.ERR_INVALID_ARG
    assert act(mode=0x80 | 1) == rq.ERR_INVALID_ARG              # unknown option bit
    assert act(n=-1) == rq.ERR_INVALID_ARG and act(d=0) == rq.ERR_INVALID_ARG
    assert act(d=60) == rq.ERR_UNSUPPORTED_SHAPE                  # not a multiple of 8
    assert act(mode=2, d=64 + 8) == rq.ERR_UNSUPPORTED_SHAPE      # not a multiple of the group
    assert act(mode=6, si=SI, d=24) == rq.ERR_UNSUPPORTED_SHAPE   # NVFP4 needs d % 16
    assert act(d=32768 + 8) == rq.ERR_UNSUPPORTED_SHAPE           # above the largest d
    assert act(n=0, gu=0, q=0, sc=0) == rq.OK
    assert act(gu=0) == rq.ERR_INVALID_ARG
    assert act(sc=0) == rq.ERR_INVALID_ARG                        # dynamic mode needs scales
    assert act(mode=0) == rq.ERR_INVALID_ARG                      # static needs scale_in
    assert act(gu=GU + 8) == rq.ERR_ALIGNMENT
    assert act(sc=SC + 2) == rq.ERR_ALIGNMENT
    assert act(q=GU + 64) == rq.ERR_ALIAS                         # codes over the input
    assert act(sc=Q + 16) == rq.ERR_ALIAS                         # scales over the codes
    if not torch.cuda.is_available():
        assert act() == rq.ERR_NO_DEVICE
        assert act(d=32768) == rq.ERR_NO_DEVICE                   # wider than the norm op allows: fine here


def test_unfused_ops_argument_errors(L):
    vp = ctypes.c_void_p
    X, R, W, Y, RO, Q, SC = 0x40000000, 0x41000000, 0x42000000, 0x43000000, 0x44000000, 0x45000000, 0x46000000

    def norm(x=X, r=R, w=W, eps=1e-6, y=Y, ro=RO, n=4, H=64, dt=0):
        return L.rmsq_fused_add_rmsnorm(vp(x) if x else None, vp(r) if r else None, vp(w) if w else None,
                                        ctypes.c_float(eps), vp(y) if y else None, vp(ro) if ro else None,
                                        n, H, dt, None)

    def qnt(y=Y, mode=1, si=0, q=Q, sc=SC, n=4, H=64, dt=0):
        return L.rmsq_quant(vp(y) if y else None, mode, vp(si) if si else None, vp(q) if q else None,
                            vp(sc) if sc else None, n, H, dt, None)

    assert norm(dt=2) == rq.ERR_INVALID_ARG
    assert norm(eps=-1.0) == rq.ERR_INVALID_ARG and norm(eps=float("nan")) == rq.ERR_INVALID_ARG
    assert norm(H=60) == rq.ERR_UNSUPPORTED_SHAPE and norm(H=16392) == rq.ERR_UNSUPPORTED_SHAPE
    assert norm(y=0) == rq.ERR_INVALID_ARG
    assert norm(ro=0) == rq.ERR_INVALID_ARG                       # residual without residual_out
    assert norm(x=X + 8) == rq.ERR_ALIGNMENT and norm(y=Y + 4) == rq.ERR_ALIGNMENT
    assert norm(y=X + 16) == rq.ERR_ALIAS                         # y over x
    assert norm(ro=W) == rq.ERR_ALIAS                             # residual_out over the weight
    assert norm(n=0, x=0, r=0, w=0, y=0, ro=0) == rq.OK
    assert qnt(dt=2) == rq.ERR_INVALID_ARG
    assert qnt(mode=7) == rq.ERR_INVALID_ARG
    assert qnt(mode=0) == rq.ERR_INVALID_ARG                      # static needs scale_in
    assert qnt(sc=0) == rq.ERR_INVALID_ARG
    assert qnt(mode=2, H=96) == rq.ERR_UNSUPPORTED_SHAPE
    assert qnt(q=Y + 64) == rq.ERR_ALIAS
    assert qnt(n=0, y=0, q=0, sc=0) == rq.OK
    if not torch.cuda.is_available():
        assert norm() == rq.ERR_NO_DEVICE
        assert norm(r=0, ro=0) == rq.ERR_NO_DEVICE                # no residual
        assert norm(ro=R) == rq.ERR_NO_DEVICE                     # in place
        assert qnt() == rq.ERR_NO_DEVICE


def test_qk_norm_rope_argument_errors(L):
    vp = ctypes.c_void_p
    Q, P_, CS, W1, W2 = 0x60000000, 0x61000000, 0x62000000, 0x63000000, 0x64000000

    def qk(qkv=Q, pos=P_, cs=CS, mp=64, qw=W1, kw=W2, eps=1e-6, n=4, nq=2, nkv=1, D=128, neox=1, dt=0, v=0):
        return L.rmsq_qk_norm_rope_ex(vp(qkv) if qkv else None, vp(pos) if pos else None,
                                      vp(cs) if cs else None, mp, vp(qw) if qw else None,
                                      vp(kw) if kw else None, ctypes.c_float(eps), n, nq, nkv, D, neox, dt,
                                      None, v)

    assert qk(v=3) == rq.ERR_INVALID_ARG and qk(v=-1) == rq.ERR_INVALID_ARG
    assert qk(dt=2) == rq.ERR_INVALID_ARG
    assert qk(neox=2) == rq.ERR_INVALID_ARG
    assert qk(nq=0, nkv=0) == rq.ERR_INVALID_ARG
    assert qk(mp=0) == rq.ERR_INVALID_ARG
    assert qk(eps=float("nan")) == rq.ERR_INVALID_ARG
    assert qk(D=96) == rq.ERR_UNSUPPORTED_SHAPE
    assert qk(nq=5000) == rq.ERR_UNSUPPORTED_SHAPE
    assert qk(qkv=0) == rq.ERR_INVALID_ARG
    assert qk(qkv=Q + 8) == rq.ERR_ALIGNMENT
    assert qk(pos=P_ + 4) == rq.ERR_ALIGNMENT
    assert qk(cs=Q + 256) == rq.ERR_ALIAS                   # table inside qkv
    assert qk(n=0, qkv=0, pos=0, cs=0, qw=0, kw=0) == rq.OK
    if not torch.cuda.is_available():
        for v in (0, 1, 2):
            assert qk(v=v) == rq.ERR_NO_DEVICE


def test_query_launch_argument_errors(L):
    out = (ctypes.c_int32 * 5)()
    assert L.rmsq_query_launch(1, 16, 4096, 1, 2, 0, out) == rq.ERR_INVALID_ARG       # dtype
    assert L.rmsq_query_launch(1, 16, 4096, 1, 0, 3, out) == rq.ERR_INVALID_ARG       # variant
    assert L.rmsq_query_launch(1, 16, 4096, 2, 0, 0, out) == rq.ERR_INVALID_ARG       # residual flag
    assert L.rmsq_query_launch(1, 16, 4096, 1, 0, 0, None) == rq.ERR_INVALID_ARG
    assert L.rmsq_query_launch(9, 16, 4096, 1, 0, 0, out) == rq.ERR_INVALID_ARG       # mode
    assert L.rmsq_query_launch(2, 16, 4000, 1, 0, 0, out) == rq.ERR_UNSUPPORTED_SHAPE  # not a multiple of 128
    for i in range(5):
        out[i] = 7
    assert L.rmsq_query_launch(1, 0, 4096, 1, 0, 0, out) == rq.OK and list(out) == [0] * 5
    if not torch.cuda.is_available():
        assert L.rmsq_query_launch(1, 16, 4096, 1, 0, 0, out) == rq.ERR_NO_DEVICE


def test_process_wide_switches(L):
    """The tuning switches only store settings: valid values are accepted,
    others rejected, and the defaults are put back."""
    assert L.rmsq_set_programmatic_launch(2) == rq.ERR_INVALID_ARG
    assert L.rmsq_set_programmatic_launch(-1) == rq.ERR_INVALID_ARG
    assert L.rmsq_set_programmatic_launch(0) == 0
    assert L.rmsq_set_programmatic_launch(1) == 0
    assert L.rmsq_set_pipeline_config(3, 0, 0, 0) == rq.ERR_INVALID_ARG
    assert L.rmsq_set_pipeline_config(0, 9, 0, 0) == rq.ERR_INVALID_ARG
    assert L.rmsq_set_pipeline_config(0, 0, 0, 3) == rq.ERR_INVALID_ARG
    assert L.rmsq_set_pipeline_config(2, 2, 1, 2) == 0
    assert L.rmsq_set_pipeline_config(0, 0, 0, 0) == 0
