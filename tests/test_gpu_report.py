"""The drift report (schema rlk_attn_cp_drift/v1) on a small workload: every
strict drift class is exactly 0.0 and the report carries the Report Contract
fields ("WS2 Attention PR5 Drift Benchmark", drift-class table and Report
Contract)."""
import numpy as np
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


def _dlogp_tol(w):
    # |d dlogp| <= |d logit_tok| + |d lse| <= 2 max_j |d logit_j|, and
    # |d logit_j| = |sum_i d x_i W_ij| <= max_i |d x_i| * sum_i |W_ij|: with
    # the output gate |d x| <= TOL_OUT, the dlogp gate is
    # 2 * TOL_OUT * max_j |W[:, j]|_1
    from tests.gpu_helpers import TOL_OUT
    return 2.0 * TOL_OUT * float(np.abs(w.astype(np.float64)).sum(axis=0).max())


def test_dlogp_of_gpu_out_matches_the_oracle():
    # the drift report's dlogp class against the oracle: the selected-token
    # log-probability of the GPU's FP32 output and of the oracle's FP64
    # output, both projected by the oracle's FP64 head, on the tiny workload
    # (all 256 rows) and on sampled rows of the varlen prefill workload
    import oracle
    from deterministic_context_attention_gb300 import synth
    from tests.gpu_helpers import device_inputs, run_fused
    from tests.test_gpu_fullsize import sample_rows
    for cfg, n_rows in ((synth.CFG_TINY, None), (synth.CFG_PREFILL, 60)):
        prob = synth.prefill_problem(**cfg)
        out, _, _ = run_fused(prob, qkv=device_inputs(prob))
        rows = np.arange(out.shape[0]) if n_rows is None else sample_rows(prob.cu_q, n_rows, 3)
        ref_out, _ = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=rows)
        w, tok = synth.lm_head(prob.hq * 128, len(rows))
        got = oracle.dlogp_f64(out[rows], w, tok)
        ref = oracle.dlogp_f64(ref_out, w, tok)
        err, tol = float(np.abs(got - ref).max()), _dlogp_tol(w)
        assert err <= tol, f"dlogp {cfg['lens']}: max |gpu - oracle| = {err:.3g} > {tol:.3g}"
