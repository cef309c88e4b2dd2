"""Pins of the CPU oracle against what the pages and mathematics fix.

Each check is chosen so that a plausible slip in the oracle (a dropped term,
a wrong sign or index, a transposed operand, a wrong causal offset, a wrong
GQA mapping) fails at least one of them.  No check retypes the oracle's own
formula: they use hand-worked closed forms (tests/golden), library routines
(scipy), the log-sum-exp decomposition identity, finite differences and
invariants.
"""
import json
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax

import oracle
from oracle import cp as ocp
from deterministic_context_attention_gb300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def small_problem(lens, hq=4, hkv=2, d=16, seed=11, kv_lens=None, block=8):
    return synth.prefill_problem(lens, hq=hq, hkv=hkv, d=d, block=block, seed=seed,
                                 kv_lens=kv_lens)


# --- closed forms ---------------------------------------------------------

def test_handworked_golden():
    cases = json.load(open(os.path.join(GOLDEN, "handworked.json")))["cases"]
    for c in cases:
        q = np.array(c["q"], np.float32)[:, None, :]
        k = np.array(c["k"], np.float32)[:, None, :]
        v = np.array(c["v"], np.float32)[:, None, :]
        n = q.shape[0]
        cu = np.array([0, n], np.int32)
        out, lse = oracle.attention_f64(q, k, v, cu, cu, c["scale"])
        tol = c.get("tol", 1e-15)
        np.testing.assert_allclose(out[:, 0, :], np.array(c["out"]), atol=tol, rtol=0, err_msg=c["name"])
        np.testing.assert_allclose(lse[:, 0], np.array(c["lse"]), atol=tol, rtol=0, err_msg=c["name"])


def test_zero_query_prefix_mean():
    # q = 0: every visible score is 0, so lse_i = ln(i+1), out_i = mean(v_0..v_i)
    p = small_problem([37])
    q = np.zeros_like(p.q)
    out, lse = oracle.attention_f64(q, p.k, p.v, p.cu_q, p.cu_k, p.scale)
    n = q.shape[0]
    np.testing.assert_allclose(lse, np.log(np.arange(1, n + 1))[:, None].repeat(p.hq, 1), atol=1e-13)
    group = p.hq // p.hkv
    for h in range(p.hq):
        pm = np.cumsum(p.v[:, h // group, :].astype(np.float64), axis=0) / np.arange(1, n + 1)[:, None]
        np.testing.assert_allclose(out[:, h, :], pm, atol=1e-13)


def test_dominant_score_selects_value():
    # one-hot keys and q_i = 64 k_i: row i scores 64 on key i and <= 0 on the
    # others, so out_i = v_i up to e^-64 weights
    n, d = 12, 8
    k = np.zeros((n, 1, d), np.float32)
    for j in range(n):
        k[j, 0, j % d] = 1.0 if j < d else -1.0
    q = 64.0 * k.copy()
    v = synth.normal_bf16(5, 3, (n, 1, d))
    cu = np.array([0, n], np.int32)
    out, lse = oracle.attention_f64(q, k, v, cu, cu, 1.0)
    for i in range(d):
        np.testing.assert_allclose(out[i, 0], v[i, 0], atol=1e-20)


def test_scipy_softmax_noncausal_and_causal():
    rng = np.random.default_rng(3)
    n, m, d = 9, 13, 6
    q = synth.bf16_round(rng.standard_normal((n, 1, d)).astype(np.float32))
    k = synth.bf16_round(rng.standard_normal((m, 1, d)).astype(np.float32))
    v = synth.bf16_round(rng.standard_normal((m, 1, d)).astype(np.float32))
    scale = 0.37
    s = scale * (q[:, 0, :].astype(np.float64) @ k[:, 0, :].astype(np.float64).T)
    out, lse = oracle.attention_f64(q, k, v, np.array([0, n], np.int32), np.array([0, m], np.int32),
                                    scale, causal=False)
    np.testing.assert_allclose(lse[:, 0], logsumexp(s, axis=1), atol=1e-13)
    np.testing.assert_allclose(out[:, 0, :], softmax(s, axis=1) @ v[:, 0, :].astype(np.float64), atol=1e-13)
    # causal, bottom-right: row i sits at position m - n + i and sees keys <= it
    out_c, lse_c = oracle.attention_f64(q, k, v, np.array([0, n], np.int32), np.array([0, m], np.int32),
                                        scale, causal=True)
    for i in range(n):
        vis = m - n + i + 1
        np.testing.assert_allclose(lse_c[i, 0], logsumexp(s[i, :vis]), atol=1e-13)
        np.testing.assert_allclose(out_c[i, 0], softmax(s[i, :vis]) @ v[:vis, 0].astype(np.float64), atol=1e-13)


def test_gqa_mapping_equals_repeated_kv_heads():
    p = small_problem([20, 7], hq=8, hkv=2)
    group = p.hq // p.hkv
    k_rep = np.repeat(p.k, group, axis=1)  # head h uses kv head h // group
    v_rep = np.repeat(p.v, group, axis=1)
    a, la = oracle.attention_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale)
    b, lb = oracle.attention_f64(p.q, k_rep, v_rep, p.cu_q, p.cu_k, p.scale)
    assert np.array_equal(a, b) and np.array_equal(la, lb)
    # and differs from the transposed mapping h % hkv
    k_bad = np.stack([p.k[:, h % p.hkv] for h in range(p.hq)], axis=1)
    c, _ = oracle.attention_f64(p.q, k_bad, v_rep, p.cu_q, p.cu_k, p.scale)
    assert not np.allclose(a, c)


def test_varlen_sequences_are_independent():
    p = small_problem([11, 30, 5])
    out, lse = oracle.attention_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale)
    for s in range(3):
        a, b = p.cu_q[s], p.cu_q[s + 1]
        o1, l1 = oracle.attention_f64(p.q[a:b], p.k[a:b], p.v[a:b], np.array([0, b - a], np.int32),
                                      np.array([0, b - a], np.int32), p.scale)
        assert np.array_equal(out[a:b], o1) and np.array_equal(lse[a:b], l1)


def test_row_subset_matches_full():
    p = small_problem([40, 9])
    out, lse = oracle.attention_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale)
    rows = np.array([48, 0, 39, 40, 17])
    o2, l2 = oracle.attention_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, rows=rows)
    assert np.array_equal(o2, out[rows]) and np.array_equal(l2, lse[rows])


# --- partial states and the merge ------------------------------------------

@pytest.mark.parametrize("block", [1, 3, 8, 64])
def test_block_states_reproduce_full_attention(block):
    # log-sum-exp decomposition: lse = log sum_b exp(lse_b),
    # out = sum_b exp(lse_b - lse) o_b, for any block size
    p = small_problem([45], block=block)
    out, lse = oracle.attention_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale)
    for t in [0, 7, 8, 31, 44]:
        for h in [0, 3]:
            o, lb = oracle.row_block_states_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, block, t, h)
            assert o.shape[0] == (t + 1 + block - 1) // block
            L = logsumexp(lb)
            np.testing.assert_allclose(L, lse[t, h], atol=1e-12)
            np.testing.assert_allclose((np.exp(lb - L)[:, None] * o).sum(0), out[t, h], atol=1e-12)


def test_block_state_of_single_key_block():
    # a block holding exactly one visible key: o_b = v_j, lse_b = s_j
    p = small_problem([10], block=4, hq=2, hkv=1, d=8)
    t = 8  # position 8: block 2 holds keys 8..11, only key 8 visible
    o, lb = oracle.row_block_states_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, 4, t, 1)
    assert o.shape[0] == 3
    np.testing.assert_array_equal(o[2], p.v[8, 0].astype(np.float64))
    s = p.scale * float(np.dot(p.q[8, 1].astype(np.float64), p.k[8, 0].astype(np.float64)))
    np.testing.assert_allclose(lb[2], s, atol=1e-15)


def tiny_states(block=64, token=255, head=5):
    p = synth.prefill_problem(**synth.CFG_TINY)
    o, lb = oracle.row_block_states_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, block, token, head)
    return p, o, lb


def test_fold_f32_close_to_fp64_truth():
    p = synth.prefill_problem(**synth.CFG_TINY)
    rows = np.array([0, 1, 63, 64, 100, 200, 255])
    out, lse = oracle.attention_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, rows=rows)
    for r, t in enumerate(rows):
        for h in range(0, 32, 7):
            o, lb = oracle.row_block_states_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, 64, t, h)
            f, fl = oracle.fold_f32(np.arange(len(lb)), o, lb)
            np.testing.assert_allclose(f, out[r, h], atol=2e-6)
            np.testing.assert_allclose(fl, lse[r, h], atol=2e-6)


def test_fold_one_state_is_identity_and_equal_lse_halves():
    o = np.array([[1.5, -2.0, 0.25]], np.float32)
    f, fl = oracle.fold_f32([4], o, np.array([0.75], np.float32))
    assert np.array_equal(f, o[0]) and fl == np.float32(0.75)
    # two states with equal lse: weights 1/2 each, lse + ln 2
    o2 = np.array([[1.0, 2.0], [3.0, -6.0]], np.float32)
    f, fl = oracle.fold_f32([0, 1], o2, np.array([1.0, 1.0], np.float32))
    np.testing.assert_allclose(f, [2.0, -2.0], atol=1e-6)
    np.testing.assert_allclose(fl, 1.0 + np.log(2.0), atol=1e-6)


def test_fold_skips_empty_state():
    o = np.array([[1.0, 1.0], [np.nan, np.nan], [3.0, 5.0]], np.float32)
    lse = np.array([0.5, -np.inf, 0.5], np.float32)
    f, fl = oracle.fold_f32([0, 1, 2], o, lse)
    np.testing.assert_allclose(f, [2.0, 3.0], atol=1e-6)


def test_reversed_and_random_arrival_equal_sorted_bitwise():
    # "merge_order_probe": reversed-arrival states vs canonical sorted merge
    for token, head in [(255, 5), (130, 0), (64, 31)]:
        _, o, lb = tiny_states(token=token, head=head)
        o32, l32 = o.astype(np.float32), lb.astype(np.float32)
        nb = len(l32)
        ref, rl = oracle.fold_f32(np.arange(nb), o32, l32)
        rev = np.arange(nb)[::-1].copy()
        f, fl = oracle.fold_f32(rev, o32[rev], l32[rev])
        assert np.array_equal(f, ref) and fl == rl
        rng = np.random.default_rng(token)
        for _ in range(5):
            perm = rng.permutation(nb)
            f, fl = oracle.fold_f32(perm, o32[perm], l32[perm])
            assert np.array_equal(f, ref) and fl == rl


def test_arrival_order_fold_is_not_canonical():
    # negative control (reduction_order = ARRIVAL): folding in arrival order
    # must differ from the canonical fold somewhere on the tiny workload
    p = synth.prefill_problem(**synth.CFG_TINY)
    differs = 0
    for token in range(192, 256, 4):
        for head in range(0, 32, 4):
            o, lb = oracle.row_block_states_f64(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, 64, token, head)
            o32, l32 = o.astype(np.float32), lb.astype(np.float32)
            rev = np.arange(len(l32))[::-1].copy()
            ref, rl = oracle.fold_f32(np.arange(len(l32)), o32, l32)
            f, fl = oracle.fold_f32(rev, o32[rev], l32[rev], arrival_order=True)
            differs += int(not (np.array_equal(f, ref) and fl == rl))
    assert differs > 0


def test_duplicate_block_index_is_rejected():
    o = np.zeros((3, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.fold_f32([0, 2, 2], o, np.zeros(3, np.float32))


# --- emulated context parallelism -----------------------------------------

@pytest.mark.parametrize("layout", [ocp.CONTIGUOUS, ocp.ZIGZAG])
@pytest.mark.parametrize("cp", [2, 4, 8])
def test_partition_covers_every_token_once(cp, layout):
    for n in [1, 7, 16, 777, 1024, 3000, 4096]:
        seen = np.zeros(n, np.int32)
        for rank, b, e in ocp.chunks(n, cp, layout):
            assert 0 <= rank < cp
            seen[b:e] += 1
        assert np.all(seen == 1)
        if layout == ocp.ZIGZAG and n >= 2 * cp:
            loads = np.zeros(cp)
            for rank, b, e in ocp.chunks(n, cp, layout):
                loads[rank] += sum(range(b + 1, e + 1))  # causal work of the rows
            assert loads.max() / loads.min() < 1.2


@pytest.mark.parametrize("layout", [ocp.CONTIGUOUS, ocp.ZIGZAG])
@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_emulated_cp_equals_cp1_bitwise(cp, layout):
    p = synth.prefill_problem(lens=[300, 129], hq=4, hkv=2, d=32, block=16, seed=7)
    rng = np.random.default_rng(cp)
    for token in [0, 15, 16, 170, 299, 300, 428]:
        for head in [0, 3]:
            ref, rl, arr1 = ocp.emulated_cp_fold(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, 16, 1,
                                                layout, token, head)
            order = rng.permutation(cp)
            out, lse, arr = ocp.emulated_cp_fold(p.q, p.k, p.v, p.cu_q, p.cu_k, p.scale, 16, cp,
                                                 layout, token, head, rank_order=order,
                                                 reverse_within_rank=True)
            assert sorted(arr) == list(range(len(arr1)))  # every block produced exactly once
            assert np.array_equal(out, ref) and lse == rl


# --- chunked replay and paged decode ----------------------------------------

def test_chunked_rows_equal_full_prefill_rows():
    full = synth.prefill_problem(lens=[50], hq=4, hkv=2, d=16, seed=9)
    out, lse = oracle.attention_f64(full.q, full.k, full.v, full.cu_q, full.cu_k, full.scale)
    for c0, c1 in [(0, 1), (1, 17), (17, 50), (49, 50)]:
        q = full.q[c0:c1]
        k = full.k[:c1]
        v = full.v[:c1]
        o, l = oracle.attention_f64(q, k, v, np.array([0, c1 - c0], np.int32),
                                    np.array([0, c1], np.int32), full.scale)
        assert np.array_equal(o, out[c0:c1]) and np.array_equal(l, lse[c0:c1])


def test_paged_decode_equals_last_prefill_row():
    dec = synth.paged_decode_problem(n=5, ctx=[1, 15, 16, 17, 70], hq=4, hkv=2, d=16,
                                     page_size=4, seed=13, spare_pages=6)
    out, lse = oracle.decode_paged_f64(dec.q, dec.k_pool, dec.v_pool, dec.page_table,
                                       dec.seqlens, dec.scale)
    for s in range(5):
        ctx = int(dec.seqlens[s])
        q = np.zeros((ctx, dec.hq, dec.d), np.float32)
        q[-1] = dec.q[s]
        cu = np.array([0, ctx], np.int32)
        ks, vs = dec.seq_kv(s)
        o, l = oracle.attention_f64(q, ks, vs, cu, cu, dec.scale, rows=np.array([ctx - 1]))
        np.testing.assert_allclose(out[s], o[0], atol=1e-14, rtol=0)
        np.testing.assert_allclose(lse[s], l[0], atol=1e-14, rtol=0)


def test_paged_decode_invariant_to_page_permutation():
    a = synth.paged_decode_problem(n=3, ctx=[33, 5, 64], hq=4, hkv=2, d=16, page_size=8, seed=21)
    out, lse = oracle.decode_paged_f64(a.q, a.k_pool, a.v_pool, a.page_table, a.seqlens, a.scale)
    perm = np.random.default_rng(2).permutation(a.k_pool.shape[0])
    inv = np.argsort(perm)
    pt = np.where(a.page_table >= 0, inv[np.maximum(a.page_table, 0)], -1).astype(np.int32)
    o2, l2 = oracle.decode_paged_f64(a.q, a.k_pool[perm], a.v_pool[perm], pt, a.seqlens, a.scale)
    assert np.array_equal(o2, out) and np.array_equal(l2, lse)


# --- backward ---------------------------------------------------------------

def _fd_problem(seed=4):
    # values on a 1/16 grid so that q +- 2^-8 is exact in float32
    rng = np.random.default_rng(seed)
    t, hq, hkv, d = 6, 4, 2, 4
    mk = lambda shape: (rng.integers(-24, 25, size=shape) / 16.0).astype(np.float32)
    return mk((t, hq, d)), mk((t, hkv, d)), mk((t, hkv, d)), mk((t, hq, d)), np.array([0, 4, 6], np.int32)


def _loss(q, k, v, dout, cu, scale):
    out, _ = oracle.attention_f64(q, k, v, cu, cu, scale)
    return float(np.sum(out * dout.astype(np.float64)))


@pytest.mark.parametrize("which", ["q", "k", "v"])
def test_backward_matches_finite_differences(which):
    q, k, v, dout, cu = _fd_problem()
    scale = 0.5
    dq, dk, dv = oracle.backward_f64(q, k, v, dout, cu, scale)
    grad = {"q": dq, "k": dk, "v": dv}[which]
    x = {"q": q, "k": k, "v": v}[which]
    worst = 0.0
    for idx in np.ndindex(x.shape):
        def f(h):
            xs = x.copy()
            xs[idx] = np.float32(x[idx] + h)
            args = {"q": q, "k": k, "v": v}
            args[which] = xs
            return _loss(args["q"], args["k"], args["v"], dout, cu, scale)
        h = 2.0 ** -8
        d1 = (f(h) - f(-h)) / (2 * h)
        d2 = (f(h / 2) - f(-h / 2)) / h
        fd = (4 * d2 - d1) / 3  # Richardson: O(h^4)
        worst = max(worst, abs(fd - grad[idx]))
    assert worst < 1e-8, worst


def test_backward_invariants():
    p = small_problem([23, 9], hq=4, hkv=2, d=8)
    zero = np.zeros_like(p.q)
    dq, dk, dv = oracle.backward_f64(p.q, p.k, p.v, zero, p.cu_q, p.scale)
    assert not dq.any() and not dk.any() and not dv.any()
    # all keys equal: softmax shifts do not move out, so dQ = 0
    k_eq = np.broadcast_to(p.k[:1], p.k.shape).copy()
    dout = synth.normal_bf16(3, synth.T_DOUT, p.q.shape)
    dq, _, _ = oracle.backward_f64(p.q, k_eq, p.v, dout, p.cu_q, p.scale)
    assert np.abs(dq).max() < 1e-12
    # dV sums P^T dout over rows: the column sums of P are what dV of a
    # dout of ones sees -- sum over keys of dV = sum over rows of dout
    dq, dk, dv = oracle.backward_f64(p.q, p.k, p.v, dout, p.cu_q, p.scale)
    group = p.hq // p.hkv
    for g in range(p.hkv):
        for s in range(2):
            a, b = p.cu_q[s], p.cu_q[s + 1]
            np.testing.assert_allclose(dv[a:b, g].sum(0),
                                       dout[a:b, g * group:(g + 1) * group].astype(np.float64).sum((0, 1)),
                                       atol=1e-11)
            # sum_j dS_ij = 0 for every row, so sum_j dK_j = scale sum_i (sum_j dS_ij) q_i = 0
            np.testing.assert_allclose(dk[a:b, g].sum(0), 0.0, atol=1e-11)


def test_backward_gqa_equals_sum_of_mha():
    p = small_problem([17], hq=4, hkv=2, d=8)
    dout = synth.normal_bf16(8, synth.T_DOUT, p.q.shape)
    dq, dk, dv = oracle.backward_f64(p.q, p.k, p.v, dout, p.cu_q, p.scale)
    group = p.hq // p.hkv
    k_rep = np.repeat(p.k, group, axis=1)
    v_rep = np.repeat(p.v, group, axis=1)
    dq2, dk2, dv2 = oracle.backward_f64(p.q, k_rep, v_rep, dout, p.cu_q, p.scale)
    np.testing.assert_allclose(dq, dq2, atol=1e-13)
    np.testing.assert_allclose(dk, dk2.reshape(dk2.shape[0], p.hkv, group, -1).sum(2), atol=1e-13)
    np.testing.assert_allclose(dv, dv2.reshape(dv2.shape[0], p.hkv, group, -1).sum(2), atol=1e-13)


def test_backward_restriction_matches_full():
    p = small_problem([12, 20], hq=4, hkv=2, d=8)
    dout = synth.normal_bf16(8, synth.T_DOUT, p.q.shape)
    dq, dk, dv = oracle.backward_f64(p.q, p.k, p.v, dout, p.cu_q, p.scale)
    dq1, dk1, dv1 = oracle.backward_f64(p.q, p.k, p.v, dout, p.cu_q, p.scale, only_seq=1, only_group=1)
    a, b = p.cu_q[1], p.cu_q[2]
    assert np.array_equal(dq1[a:b, 2:4], dq[a:b, 2:4])
    assert np.array_equal(dk1[a:b, 1], dk[a:b, 1]) and np.array_equal(dv1[a:b, 1], dv[a:b, 1])
    assert np.isnan(dq1[:a]).all()


# --- RoPE -------------------------------------------------------------------

def test_rope_handworked_golden():
    cases = json.load(open(os.path.join(GOLDEN, "rope_handworked.json")))["cases"]
    for c in cases:
        d = c["d"]
        x = np.zeros((1, 1, d), np.float32)
        for i, v in c["x"].items():
            x[0, 0, int(i)] = v
        want = np.zeros(d, np.float32)
        for i, v in c["y"].items():
            want[int(i)] = v
        y = oracle.rope_f32(x, [c["pos"]], c["theta"])
        np.testing.assert_array_equal(y[0, 0], want, err_msg=c["name"])


def _bf16_round(a):
    b = np.ascontiguousarray(a, np.float32).view(np.uint32).astype(np.uint64)
    b = (b + 0x7FFF + ((b >> 16) & 1)) & 0xFFFF0000
    return b.astype(np.uint32).view(np.float32)


def _rope_rows(t, h, d, seed):
    rng = np.random.default_rng(seed)
    return _bf16_round(rng.standard_normal((t, h, d)).astype(np.float32))


def test_rope_exact_equals_complex_rotation():
    # the rotation of pair (i, i + D/2) is multiplication of x_i + j x_{i+D/2}
    # by exp(j * p * theta^(-2i/D)): a second formulation, in numpy complex
    t, h, d, theta = 37, 3, 16, 1e4
    x = _rope_rows(t, h, d, 1)
    pos = np.random.default_rng(2).integers(0, 50000, t).astype(np.int32)
    y = oracle.rope_f64(x, pos, theta)
    f = theta ** (-np.arange(d // 2) * 2.0 / d)
    z = (x[..., : d // 2] + 1j * x[..., d // 2:].astype(np.float64)) * np.exp(1j * pos[:, None, None] * f[None, None, :])
    np.testing.assert_allclose(y[..., : d // 2], z.real, rtol=0, atol=1e-12)
    np.testing.assert_allclose(y[..., d // 2:], z.imag, rtol=0, atol=1e-12)


def test_rope_exact_relative_position_property():
    # <R(m) q, R(n) k> depends on m - n only
    d, theta = 128, 1e6
    q = _rope_rows(1, 1, d, 3)
    k = _rope_rows(1, 1, d, 4)
    for m, n, s in [(5, 2, 1000), (0, 0, 31), (4000, 17, 12345)]:
        a = np.dot(oracle.rope_f64(q, [m], theta)[0, 0], oracle.rope_f64(k, [n], theta)[0, 0])
        b = np.dot(oracle.rope_f64(q, [m + s], theta)[0, 0], oracle.rope_f64(k, [n + s], theta)[0, 0])
        assert abs(a - b) <= 1e-9 * (1 + abs(a))


@pytest.mark.parametrize("theta", [1e6, 1e4])
def test_rope_f32_is_bf16_rounding_of_exact_rotation(theta):
    # the canonical FP32 form differs from the exact rotation only by the
    # FP32 steps (a few 2^-24 relative) before the one BF16 rounding: within
    # one BF16 ulp everywhere, and equal to bf16_rn(exact) almost everywhere
    t, h, d = 300, 4, 128
    x = _rope_rows(t, h, d, 5)
    pos = np.random.default_rng(6).integers(0, 40000, t).astype(np.int32)
    y32 = oracle.rope_f32(x, pos, theta).astype(np.float64)
    y64 = oracle.rope_f64(x, pos, theta)
    ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(y64), 1e-30))) - 7)
    assert np.all(np.abs(y32 - y64) <= ulp + 1e-30)
    same = np.mean(y32 == _bf16_round(y64.astype(np.float32)).astype(np.float64))
    assert same > 0.999
    assert np.all(_bf16_round(y32.astype(np.float32)) == y32.astype(np.float32))  # results are BF16 values


def test_rope_position_zero_is_identity_and_rows_are_independent():
    t, h, d = 9, 2, 128
    x = _rope_rows(t, h, d, 7)
    np.testing.assert_array_equal(oracle.rope_f32(x, np.zeros(t, np.int32), 1e6), x)
    pos = np.arange(t, dtype=np.int32) * 100
    full = oracle.rope_f32(x, pos, 1e6)
    for i in (0, 4, 8):
        np.testing.assert_array_equal(oracle.rope_f32(x[i:i + 1], pos[i:i + 1], 1e6), full[i:i + 1])
