"""Pins of the oracle's selected-token log-probability (oracle.dlogp_f64):
the dlogp drift class of the drift report ("WS2 Attention PR5 Drift
Benchmark", the --include-dlogp paragraph: a seeded synthetic FP32 lm_head
over the attention output and the active token's selected log-probability;
"[WS2][Attention] H100 validation and reproduction guide", Status: dlogp max
abs 0.0).  Each pin is fixed by the mathematics, not by the code: hand-worked
closed forms (tests/golden/dlogp_handworked.json), scipy's log_softmax, and
the invariance of a log-softmax to a common shift of the logits.  The
report's own FP32 projection is then checked against the pinned oracle."""
import json
import os

import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from deterministic_context_attention_gb300.report import _dlogp

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dlogp_handworked.json")


@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_dlogp_handworked(case):
    got = oracle.dlogp_f64(np.array(case["x"]), np.array(case["w"]), np.array(case["tok"]))
    np.testing.assert_allclose(got, case["dlogp"], rtol=0, atol=1e-14)


def test_dlogp_zero_outputs_is_minus_log_vocab():
    for vocab in (2, 7, 512):
        w, tok = synth.lm_head(96, 5, vocab, seed=3)
        got = oracle.dlogp_f64(np.zeros((5, 96)), w, tok)
        np.testing.assert_allclose(got, -np.log(vocab), rtol=0, atol=1e-14)


def test_dlogp_matches_scipy_log_softmax():
    scipy_special = pytest.importorskip("scipy.special")
    out = np.random.default_rng(1).standard_normal((9, 4, 128))
    w, tok = synth.lm_head(512, 9, 300, seed=11)
    logits = out.reshape(9, -1) @ w.astype(np.float64)
    ref = scipy_special.log_softmax(logits, axis=1)[np.arange(9), tok]
    np.testing.assert_allclose(oracle.dlogp_f64(out, w, tok), ref, rtol=0, atol=1e-12)


def test_dlogp_shift_invariance_and_token_selection():
    # a constant added to every logit (an extra input 1 with a constant head
    # row) leaves dlogp unchanged; the selected token's logit, not another's,
    # enters (a wrong index would move the value)
    rng = np.random.default_rng(5)
    out = rng.standard_normal((6, 64))
    w, tok = synth.lm_head(64, 6, 40, seed=9)
    base = oracle.dlogp_f64(out, w, tok)
    out1 = np.concatenate([out, np.ones((6, 1))], axis=1)
    w1 = np.concatenate([w.astype(np.float64), np.full((1, 40), 12.5)], axis=0)
    np.testing.assert_allclose(oracle.dlogp_f64(out1, w1, tok), base, rtol=0, atol=1e-12)
    other = (tok + 1) % 40
    assert np.all(np.abs(oracle.dlogp_f64(out, w, other) - base) > 0)
    assert np.all(base < 0)


def test_report_fp32_dlogp_agrees_with_the_oracle():
    # the report's projection (FP32 numpy, the same for every path compared)
    # is the oracle's quantity up to FP32 rounding
    out = np.random.default_rng(2).standard_normal((9, 4, 128)).astype(np.float32)
    w, tok = synth.lm_head(512, 9)
    assert np.max(np.abs(_dlogp(out) - oracle.dlogp_f64(out, w, tok))) < 1e-4


def test_report_dlogp_deterministic_and_sensitive():
    out = np.random.default_rng(2).standard_normal((6, 8, 128)).astype(np.float32)
    a = _dlogp(out)
    assert np.array_equal(a, _dlogp(out.copy()))
    moved = out.copy()
    moved[3, 2, 17] += 1e-3
    d = np.abs(_dlogp(moved) - a)
    assert d[3] > 0 and np.all(np.delete(d, 3) == 0)
