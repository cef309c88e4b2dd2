"""The drift report's active-token log-probability (a seeded synthetic FP32
lm_head over every head's output of a row; "[WS2][Attention] H100 validation
and reproduction guide", Status: Out/LSE/dlogp max abs 0.0): it is the log of
the softmax over the projected logits at the selected token, deterministic,
and it moves when an output element moves."""
import numpy as np

from deterministic_context_attention_gb300.report import _dlogp


def _reference_fp64(out, vocab=512, seed=7):
    rows = out.shape[0]
    x = out.reshape(rows, -1).astype(np.float64)
    rng = np.random.default_rng([seed, x.shape[1], vocab])
    w = (rng.standard_normal((x.shape[1], vocab)) / np.sqrt(x.shape[1])).astype(np.float32).astype(np.float64)
    tok = rng.integers(0, vocab, size=rows)
    logits = x @ w
    m = logits.max(axis=1, keepdims=True)
    logp = logits - (m + np.log(np.exp(logits - m).sum(axis=1, keepdims=True)))
    return logp[np.arange(rows), tok]


def test_dlogp_is_the_log_softmax_at_the_selected_token():
    out = np.random.default_rng(1).standard_normal((9, 4, 128)).astype(np.float32)
    got = _dlogp(out)
    ref = _reference_fp64(out)
    assert np.max(np.abs(got - ref)) < 1e-4
    assert np.all(got < 0)  # a log-probability


def test_dlogp_deterministic_and_sensitive():
    out = np.random.default_rng(2).standard_normal((6, 8, 128)).astype(np.float32)
    a = _dlogp(out)
    assert np.array_equal(a, _dlogp(out.copy()))
    moved = out.copy()
    moved[3, 2, 17] += 1e-3
    d = np.abs(_dlogp(moved) - a)
    assert d[3] > 0 and np.all(np.delete(d, 3) == 0)
