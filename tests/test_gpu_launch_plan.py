"""The pipelined kernel's launch plan as the library reports it
(rmsq_query_launch) and parity on the shapes that take the many-rows plan.

With at least 8 rows per CTA of the persistent grid the library switches to
a one-stage ring and more chunks per thread (4 with a residual above hidden
2048, 8 without from hidden 4096); the arithmetic is the same in every plan
(vLLM docs "Fusion torch.compile passes", section "RMSNorm + Quantization
(fuse_norm_quant)"), so every plan must give the oracle's results bit for
bit, including a ragged last wave of rows."""
import pytest
import torch

import _parity as P
import residual_add_rmsnorm_rmsq_gb300 as rq
import rmsq_inputs as ri

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib(rmsq_gpu):
    return rmsq_gpu


def many_rows(mode, hidden, residual):
    """The plan of the many-rows case for this shape: the query at a batch
    large enough to take it."""
    return rq.query_launch(mode, 1 << 20, hidden, residual)


def test_plans_follow_rows_per_cta():
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # DeepSeek-V3 layer, 8192 x 7168 with a residual: many rows per CTA
    p = rq.query_launch("fp8_group128_row", 8192, 7168, True)
    assert p["pipelined"] and p["chunks_per_thread"] == 4 and p["stages"] == 1
    assert 8192 >= 8 * p["ctas"] and p["threads"] == 224
    # Llama layer of 4096 rows: few rows per CTA, the default two-chunk, two-stage plan
    p = rq.query_launch("fp8_per_token", 4096, 4096, True)
    assert p["pipelined"] and p["chunks_per_thread"] == 2 and p["stages"] == 2
    assert 4096 < 8 * many_rows("fp8_per_token", 4096, True)["ctas"]
    # without a residual: eight chunks per thread from hidden 4096 when rows are many
    p = many_rows("fp8_per_token", 4096, False)
    assert p["chunks_per_thread"] == 8 and p["stages"] == 1
    assert many_rows("fp8_per_token", 2048, False)["chunks_per_thread"] == 4
    assert many_rows("nvfp4", 2048, True)["chunks_per_thread"] == 2
    # below 4 rows per SM the direct kernel, one CTA per row
    p = rq.query_launch("fp8_per_token", 4 * sms - 1, 4096, True)
    assert not p["pipelined"] and p["ctas"] == 4 * sms - 1 and p["stages"] == 0
    assert rq.query_launch("fp8_per_token", 0, 4096, True) == {"pipelined": False, "chunks_per_thread": 0,
                                                               "stages": 0, "ctas": 0, "threads": 0}
    # a tuned plan stays as tuned
    rq.set_pipeline_config(2, 2, 0, 0)
    try:
        p = rq.query_launch("fp8_group128_row", 8192, 7168, True)
    finally:
        rq.set_pipeline_config(0, 0, 0, 0)
    assert p["chunks_per_thread"] == 2 and p["stages"] == 2


@pytest.mark.parametrize("mode,hidden,residual", [("fp8_group128_row", 5120, True),
                                                  ("fp8_per_token", 8192, True),
                                                  ("nvfp4", 2048, True),
                                                  ("fp8_per_token", 4096, False),
                                                  ("fp8_group64_col", 2048, False)])
def test_many_rows_plan_parity(mode, hidden, residual):
    p = many_rows(mode, hidden, residual)
    n = 8 * p["ctas"] + 37            # the many-rows plan, and a ragged last wave
    assert rq.query_launch(mode, n, hidden, residual) == {**p, "ctas": p["ctas"]}
    wl = ri.make_workload(f"plan_{hidden}_{int(residual)}", n, hidden, res_sigma=1.5, residual=residual,
                          static_scale=0.05, seed=hidden + n)
    P.check(wl, mode, variants=("auto",), label=f"many-rows plan {mode} {hidden} res={residual}")
