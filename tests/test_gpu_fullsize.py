"""Parity and bit invariance at the full workload sizes, in the launch
configuration bench.py times, on sampled outputs the oracle computes row by
row:
  * varlen prefill {4096, 3000, 1024, 777}, Hq=32/Hkv=8, RoPE, KV block 128:
    oracle rows; logical CP 2/4/8 zigzag (fused row ownership and states +
    merge in permuted arrival) and batch order bitwise equal to CP=1;
  * chunked replay, Hq=16/Hkv=4, 2 x 8192: chunks of 2048, 512 and 1 bitwise
    equal to the full prefill;
  * paged decode, 64 sequences, ctx ~ U[512, 32768], 16-token pages in a
    permuted pool: oracle sequences, last prefill row bitwise, page
    permutation and batch subset bitwise.
("[WS2][Attention] H100 validation and reproduction guide", Status and
Acceptance: strict out/LSE max abs 0.0 across ranks, decode/prefill.)"""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import (assert_bitwise, assert_forward_parity, device_inputs, run_fused,
                               run_states_merge)

pytestmark = pytest.mark.gpu


def sample_rows(cu, n_random, seed):
    rows = set()
    for s in range(len(cu) - 1):
        a, b = int(cu[s]), int(cu[s + 1])
        rows.update([a, a + 1, min(a + 127, b - 1), min(a + 128, b - 1), b - 1, b - 2])
    rng = np.random.default_rng(seed)
    rows.update(rng.integers(0, int(cu[-1]), size=n_random).tolist())
    return np.array(sorted(r for r in rows if 0 <= r < cu[-1]), np.int64)


@pytest.fixture(scope="module")
def prefill_cfg():
    prob = synth.prefill_problem(**synth.CFG_PREFILL)
    return prob, device_inputs(prob)


@pytest.fixture(scope="module")
def prefill_base(prefill_cfg):
    prob, qkv = prefill_cfg
    return run_fused(prob, qkv=qkv)


def test_prefill_fullsize_parity(prefill_cfg, prefill_base):
    prob, _ = prefill_cfg
    rows = sample_rows(prob.cu_q, 80, 1)
    ref_out, ref_lse = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=rows)
    out, outb, lse = prefill_base
    assert_forward_parity(out[rows], outb[rows], lse[rows], ref_out, ref_lse, "prefill full size")


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_prefill_fullsize_cp_invariance(prefill_cfg, prefill_base, cp):
    prob, qkv = prefill_cfg
    ranks = list(np.random.default_rng(10 + cp).permutation(cp))
    assert_bitwise(run_fused(prob, cp=cp, layout=1, ranks=ranks, qkv=qkv), prefill_base, f"fused CP={cp}")
    if cp == 8:
        assert_bitwise(run_states_merge(prob, cp=cp, layout=1, rank_order=ranks, shuffle_seed=cp, qkv=qkv),
                       prefill_base, f"states+merge CP={cp}")


def test_prefill_fullsize_batch_order(prefill_cfg, prefill_base):
    prob, _ = prefill_cfg
    order = [2, 0, 3, 1]
    perm = synth.permute_batch(prob, order)
    got = run_fused(perm)
    for new_s, old_s in enumerate(order):
        a, b = perm.cu_q[new_s], perm.cu_q[new_s + 1]
        c, d = prob.cu_q[old_s], prob.cu_q[old_s + 1]
        assert_bitwise(tuple(x[a:b] for x in got), tuple(x[c:d] for x in prefill_base), f"sequence {old_s}")


# ---------------------------------------------------------------- chunked replay, TP=2 shard
@pytest.fixture(scope="module")
def chunked_cfg():
    cfg = dict(synth.CFG_CHUNKED)
    prob = synth.prefill_problem(**cfg)
    return prob, device_inputs(prob)


@pytest.fixture(scope="module")
def chunked_base(chunked_cfg):
    prob, qkv = chunked_cfg
    return run_fused(prob, qkv=qkv)


def test_chunked_fullsize_parity(chunked_cfg, chunked_base):
    prob, _ = chunked_cfg
    rows = sample_rows(prob.cu_q, 40, 2)
    ref_out, ref_lse = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=rows)
    out, outb, lse = chunked_base
    assert_forward_parity(out[rows], outb[rows], lse[rows], ref_out, ref_lse, "chunked config full prefill")


@pytest.mark.parametrize("chunk", [2048, 512, 1])
def test_chunked_fullsize_replay_bitwise(chunked_cfg, chunked_base, chunk):
    import torch
    from tests.gpu_helpers import empty_outputs, lib, params_of, to_np
    prob, (q, k, v) = chunked_cfg
    rlk = lib()
    out, outb, lse = empty_outputs(torch, q.shape[0], prob.hq)
    p = params_of(prob)
    p.num_seqs = 1
    for s in range(2):
        q0, q1, k0 = int(prob.cu_q[s]), int(prob.cu_q[s + 1]), int(prob.cu_k[s])
        for c0 in range(0, q1 - q0, chunk):
            c1 = min(c0 + chunk, q1 - q0)
            rlk.rlk_attn_prefill(p, q[q0 + c0:q0 + c1], k[k0:k0 + c1], v[k0:k0 + c1], [0, c1 - c0], [0, c1], -1,
                                 out[q0 + c0:q0 + c1], outb[q0 + c0:q0 + c1], lse[q0 + c0:q0 + c1])
    rlk.rlk_attn_check_device_error()
    assert_bitwise(to_np(out, outb, lse), chunked_base, f"chunk {chunk}")


# ---------------------------------------------------------------- paged decode
@pytest.fixture(scope="module")
def decode_cfg():
    return synth.paged_decode_problem(**synth.CFG_DECODE)


@pytest.fixture(scope="module")
def decode_base(decode_cfg):
    from tests.test_gpu_decode import run_decode
    return run_decode(decode_cfg)


def test_decode_fullsize_parity(decode_cfg, decode_base):
    dec = decode_cfg
    seqs = [int(np.argmax(dec.seqlens)), int(np.argmin(dec.seqlens)), 0, 17, 40, 63]
    out, outb, lse = decode_base
    for s in seqs:
        ks, vs = dec.seq_kv(s)
        ctx = int(dec.seqlens[s])
        q = np.zeros((ctx, dec.hq, 128), np.float32)
        q[-1] = dec.q[s]
        cu = np.array([0, ctx], np.int32)
        ro, rl = oracle.attention_f64(q, ks, vs, cu, cu, dec.scale, rows=np.array([ctx - 1]))
        assert_forward_parity(out[s:s + 1], outb[s:s + 1], lse[s:s + 1], ro, rl, f"decode seq {s} ctx {ctx}")


def test_decode_fullsize_equals_prefill_last_row(decode_cfg, decode_base):
    dec = decode_cfg
    out, outb, lse = decode_base
    for s in [int(np.argmax(dec.seqlens)), 5]:
        ks, vs = dec.seq_kv(s)
        ctx = int(dec.seqlens[s])
        q1 = dec.q[s:s + 1]
        prob = synth.Prefill(q1, ks, vs, np.array([0, 1], np.int32), np.array([0, ctx], np.int32), dec.hq,
                             dec.hkv, 128, dec.scale, 128)
        po, pb, pl = run_fused(prob)
        assert_bitwise((out[s], outb[s], lse[s]), (po[0], pb[0], pl[0]), f"sequence {s}")


def test_decode_fullsize_page_permutation_and_subset(decode_cfg, decode_base):
    from tests.test_gpu_decode import run_decode
    dec = decode_cfg
    n_pages = dec.k_bits.shape[0]
    perm = np.random.default_rng(9).permutation(n_pages)
    inv = np.argsort(perm)
    pt = np.where(dec.page_table >= 0, inv[np.maximum(dec.page_table, 0)], -1).astype(np.int32)
    moved = run_decode(dec, page_table=pt, k_bits=dec.k_bits[perm], v_bits=dec.v_bits[perm])
    assert_bitwise(moved, decode_base, "page permutation")
    subset = [63, 1, 30, 2]
    assert_bitwise(run_decode(dec, seqs=subset), tuple(x[subset] for x in decode_base), "batch subset")
