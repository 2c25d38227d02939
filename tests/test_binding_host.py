"""Host-side checks of the Python binding (no GPU needed, no kernel runs):
every wrapper rejects what the C ABI cannot express (a dtype other than
bf16 / fp16, strided tensors, malformed shapes or names) before it calls the
library, and the names map onto the header's enum values."""
import pytest
import torch

import residual_add_rmsnorm_rmsq_gb300 as rq


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from residual_add_rmsnorm_rmsq_gb300 import _build
    _build.build()
    return rq.load()


def _bf(*shape):
    return torch.zeros(*shape, dtype=torch.bfloat16)


def test_mode_and_variant_names():
    assert [rq.mode_code(m) for m in ("fp8_static", "fp8_per_token", "fp8_group128_row", "fp8_group128_col",
                                      "fp8_group64_row", "fp8_group64_col", "nvfp4")] == list(range(7))
    assert rq.mode_code("fp8_group128_col+e8m0+tma") == 3 | 0x10 | 0x20
    assert rq.mode_code("fp8_per_token+e8m0") == 1 | 0x10
    assert rq.mode_code("fp8_group64_col+ue8m0+tma") == 5 | 0x40 | 0x20
    assert rq.VARIANTS == {"auto": 0, "direct": 1, "pipelined": 2}
    with pytest.raises(ValueError):
        rq.mode_code("fp8_group32_row")
    with pytest.raises(ValueError):
        rq.mode_code("fp8_per_token+bogus")


def test_norm_quant_rejects_dtype_and_strides():
    w = _bf(64)
    with pytest.raises(TypeError):
        rq.fused_add_rmsnorm_quant(torch.zeros(4, 64), None, w, 1e-6, "fp8_per_token")
    with pytest.raises(ValueError):
        rq.fused_add_rmsnorm_quant(_bf(64, 4).t(), None, w, 1e-6, "fp8_per_token")
    with pytest.raises(ValueError):
        rq.fused_add_rmsnorm_nvfp4_dynamic(_bf(4, 128)[:, ::2], None, w, 1e-6)


def test_unfused_ops_reject_dtype_and_strides():
    w = _bf(64)
    with pytest.raises(TypeError):
        rq.fused_add_rmsnorm(torch.zeros(4, 64, dtype=torch.float16).float(), None, w, 1e-6)
    with pytest.raises(ValueError):
        rq.fused_add_rmsnorm(_bf(64, 4).t(), None, w, 1e-6)
    with pytest.raises(TypeError):
        rq.quant(torch.zeros(4, 64), "fp8_per_token")
    with pytest.raises(ValueError):
        rq.quant(_bf(4, 128)[:, ::2], "fp8_per_token")


def test_silu_mul_rejects_odd_width_dtype_and_strides():
    with pytest.raises(ValueError):
        rq.silu_mul_quant(_bf(4, 66 + 1), "fp8_static")
    with pytest.raises(TypeError):
        rq.silu_mul_quant(torch.zeros(4, 128), "fp8_static")
    with pytest.raises(ValueError):
        rq.silu_mul_quant(_bf(128, 4).t(), "fp8_static")


def test_qk_norm_rope_rejects_dtypes_and_strides():
    qkv, w = _bf(4, 4 * 128), _bf(128)
    pos = torch.zeros(4, dtype=torch.int64)
    cs = torch.zeros(16, 128, dtype=torch.float32)
    with pytest.raises(TypeError):
        rq.qk_norm_rope(qkv.float(), pos, cs, w, w, 1e-6, 2, 1, 128)
    with pytest.raises(TypeError):
        rq.qk_norm_rope(qkv, pos.int(), cs, w, w, 1e-6, 2, 1, 128)
    with pytest.raises(TypeError):
        rq.qk_norm_rope(qkv, pos, cs.double(), w, w, 1e-6, 2, 1, 128)
    with pytest.raises(ValueError):
        rq.qk_norm_rope(_bf(4 * 128, 4).t(), pos, cs, w, w, 1e-6, 2, 1, 128)
    with pytest.raises(ValueError):
        rq.qk_norm_rope(qkv, pos, cs, w, w, 1e-6, 2, 1, 128, variant="fast")
    with pytest.raises(ValueError):
        rq.fused_add_rmsnorm_quant(_bf(4, 64), None, _bf(64), 1e-6, "fp8_per_token", variant="fast")
    with pytest.raises(ValueError):
        rq.fused_add_rmsnorm_nvfp4_dynamic(_bf(4, 64), None, _bf(64), 1e-6, variant="fast")


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-device path")
def test_valid_calls_without_a_device_report_no_device():
    """Well-formed calls reach the library, which answers that there is no
    device (there is no CPU fallback)."""
    qkv, w = _bf(4, 4 * 128), _bf(128)
    pos = torch.zeros(4, dtype=torch.int64)
    cs = torch.zeros(16, 128, dtype=torch.float32)
    # stream 0 (the legacy default stream) as a raw handle: asking torch for
    # its current stream needs a driver
    with pytest.raises(rq.RmsqError) as ei:
        rq.qk_norm_rope(qkv, pos, cs, w, w, 1e-6, 2, 1, 128, stream=0)
    assert ei.value.status == rq.ERR_NO_DEVICE
    with pytest.raises(rq.RmsqError) as ei:
        rq.fused_add_rmsnorm_quant(_bf(4, 64), _bf(4, 64), _bf(64), 1e-6, "fp8_per_token", stream=0)
    assert ei.value.status == rq.ERR_NO_DEVICE
