"""GPU parity and bit-invariance of the forward path (fused prefill, states +
merge, chunked replay) against the oracle.

Tolerances ("Against the oracle"): |out_f32 - oracle| <= 2e-5,
|lse - oracle| <= 1e-5, BF16 out within 1 ulp of the oracle rounded.  Bit
invariance: the pages' strict 'max abs 0.0' claims ("[WS2][Attention] H100
validation and reproduction guide", Status / Acceptance;
"WS2 Attention PR5 Drift Benchmark", drift-class table: cp_merge_fp32,
merge_order_probe)."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import (assert_bitwise, assert_forward_parity, device_inputs, run_fused,
                               run_states_merge)

pytestmark = pytest.mark.gpu


def oracle_full(prob, rows=None):
    return oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=rows)


# ---------------------------------------------------------------- tiny config
@pytest.fixture(scope="module")
def tiny():
    return synth.prefill_problem(**synth.CFG_TINY)


def test_tiny_fused_parity(tiny):
    out, outb, lse = run_fused(tiny)
    ref_out, ref_lse = oracle_full(tiny)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, "tiny fused")


def test_tiny_states_merge_cp2_bitwise_equals_fused(tiny):
    fused = run_fused(tiny)
    # CP=2 contiguous halves; rank 1 launched and arriving first, slabs shuffled
    sm = run_states_merge(tiny, cp=2, layout=0, rank_order=[1, 0], shuffle_seed=5)
    assert_bitwise(sm, fused, "states+merge CP=2 vs fused CP=1")
    ref_out, ref_lse = oracle_full(tiny)
    assert_forward_parity(*sm, ref_out, ref_lse, "tiny merge")


def test_tiny_fused_per_rank_rows_bitwise(tiny):
    fused = run_fused(tiny)
    per_rank = run_fused(tiny, cp=2, layout=0, ranks=[1, 0])
    assert_bitwise(per_rank, fused, "fused CP=2 row ownership")


def test_repeat_runs_bitwise(tiny):
    a = run_fused(tiny)
    b = run_fused(tiny)
    assert_bitwise(a, b, "repeat")


# ---------------------------------------------------------------- medium ragged
@pytest.fixture(scope="module")
def medium():
    return synth.prefill_problem(lens=[300, 129, 1000, 17, 1], hq=32, hkv=8, block=128, seed=21, rope=True)


def test_medium_parity(medium):
    out, outb, lse = run_fused(medium)
    ref_out, ref_lse = oracle_full(medium)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, "medium fused")


@pytest.mark.parametrize("cp", [2, 4, 8])
def test_medium_cp_invariance(medium, cp):
    torch = pytest.importorskip("torch")
    qkv = device_inputs(medium)
    base = run_fused(medium, qkv=qkv)
    ranks = list(np.random.default_rng(cp).permutation(cp))
    assert_bitwise(run_fused(medium, cp=cp, layout=1, ranks=ranks, qkv=qkv), base, f"fused zigzag CP={cp}")
    assert_bitwise(run_states_merge(medium, cp=cp, layout=1, rank_order=ranks[::-1], shuffle_seed=cp, qkv=qkv),
                   base, f"states+merge zigzag CP={cp}")
    assert_bitwise(run_states_merge(medium, cp=cp, layout=0, rank_order=ranks, qkv=qkv), base,
                   f"states+merge contiguous CP={cp}")
    del torch


def test_medium_block64_parity():
    prob = synth.prefill_problem(lens=[200, 65, 64, 63], hq=8, hkv=2, block=64, seed=8)
    out, outb, lse = run_fused(prob)
    ref_out, ref_lse = oracle_full(prob)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, "block 64")
    assert_bitwise(run_states_merge(prob, cp=4, layout=1, rank_order=[3, 1, 0, 2], shuffle_seed=1),
                   (out, outb, lse), "block 64 states+merge")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (16, 2), (12, 4)])
def test_group_sizes_parity(hq, hkv):
    # groups of 1, 8 and 3 query heads per KV head (the items are (tile,
    # query head) pairs and K/V is read per KV head): oracle parity, and the
    # states + merge path equal bit for bit
    prob = synth.prefill_problem(lens=[257, 128, 1, 700], hq=hq, hkv=hkv, block=128, seed=16)
    out, outb, lse = run_fused(prob)
    ref_out, ref_lse = oracle_full(prob)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, f"hq{hq}/hkv{hkv}")
    assert_bitwise(run_states_merge(prob, cp=2, layout=1, rank_order=[1, 0], shuffle_seed=2),
                   (out, outb, lse), f"hq{hq}/hkv{hkv} states+merge")


def test_batch_order_invariance(medium):
    base = run_fused(medium)
    order = [3, 0, 4, 2, 1]
    perm = synth.permute_batch(medium, order)
    got = run_fused(perm)
    # undo the permutation sequence by sequence
    for new_s, old_s in enumerate(order):
        a, b = perm.cu_q[new_s], perm.cu_q[new_s + 1]
        c, d = medium.cu_q[old_s], medium.cu_q[old_s + 1]
        assert_bitwise(tuple(x[a:b] for x in got), tuple(x[c:d] for x in base), f"sequence {old_s}")
    # batch subset: one sequence alone
    single = synth.Prefill(medium.q[300:429], medium.k[300:429], medium.v[300:429],
                           np.array([0, 129], np.int32), np.array([0, 129], np.int32), 32, 8, 128,
                           medium.scale, 128)
    assert_bitwise(run_fused(single), tuple(x[300:429] for x in base), "batch subset")


# ---------------------------------------------------------------- chunked replay
def chunked_run(prob, chunk):
    """Replay each sequence in chunks of ``chunk`` queries against the KV
    cache up to the chunk's end; returns outputs in full-prefill layout."""
    import torch
    from tests.gpu_helpers import empty_outputs, lib, params_of, to_np
    rlk = lib()
    q, k, v = device_inputs(prob)
    out, outb, lse = empty_outputs(torch, q.shape[0], prob.hq)
    p = params_of(prob)
    p.num_seqs = 1
    for s in range(len(prob.cu_q) - 1):
        q0, q1 = int(prob.cu_q[s]), int(prob.cu_q[s + 1])
        k0 = int(prob.cu_k[s])
        for c0 in range(0, q1 - q0, chunk):
            c1 = min(c0 + chunk, q1 - q0)
            rlk.rlk_attn_prefill(p, q[q0 + c0:q0 + c1], k[k0:k0 + c1], v[k0:k0 + c1], [0, c1 - c0], [0, c1], -1,
                                 out[q0 + c0:q0 + c1], outb[q0 + c0:q0 + c1], lse[q0 + c0:q0 + c1])
    rlk.rlk_attn_check_device_error()
    return to_np(out, outb, lse)


@pytest.mark.parametrize("chunk", [1, 7, 128, 200, 512])
def test_chunked_replay_bitwise_small(chunk):
    prob = synth.prefill_problem(lens=[700, 300], hq=16, hkv=4, block=128, seed=2)
    base = run_fused(prob)
    assert_bitwise(chunked_run(prob, chunk), base, f"chunk {chunk}")
