"""The drift report (schema rlk_attn_cp_drift/v1) on a small workload: every
strict drift class is exactly 0.0 and the report carries the Report Contract
fields ("WS2 Attention PR5 Drift Benchmark", drift-class table and Report
Contract)."""
import pytest

pytestmark = pytest.mark.gpu


def test_small_drift_report_is_strictly_zero():
    from tests.gpu_helpers import torch_cuda
    torch_cuda()
    from deterministic_context_attention_gb300.report import drift_report
    rep = drift_report(lens=(300, 129, 1000, 17), cp_sizes=(2, 4), chunk_sizes=(7, 200), backward_lens=(300, 129),
                       backward_cp=(2,))
    assert rep["merge_order"] == "global_block_index" and rep["downcast_at"] == "final_write"
    assert rep["passed"], rep["strict_max_abs"]
    modes = {c["mode"] for c in rep["cases"]}
    assert modes == {"full_prefill", "chunked_prefill", "backward"}
    for c in rep["cases"]:
        if c["mode"] == "full_prefill":
            assert 0.0 < c["drift"]["dtype_path_vs_fp32"] < 0.1
            assert len(c["per_logical_cp_rank"]) == c["topology"]["cp"]
            assert len(c["block_manifest_hash"]) == 16
