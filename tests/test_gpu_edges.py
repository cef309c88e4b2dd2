"""GPU edge cases of the hot path: empty and one-token sequences inside a
varlen batch, the largest batch one call takes (128 sequences), a query
chunk of length 0, and one very long decode context (131,072 tokens: 1024
KV blocks, page ids over sixteen 512-page windows) -- each against the
oracle and, where the pages fix an invariance, bit for bit ("[WS2][Attention]
H100 validation and reproduction guide", Status and Acceptance: batch
invariance, strict decode/prefill identity)."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import (assert_bitwise, assert_forward_parity, empty_outputs, lib, run_fused,
                               run_states_merge, torch_cuda)

pytestmark = pytest.mark.gpu


def test_prefill_empty_and_one_token_sequences():
    # sequences of 0 tokens pack to nothing, so the batch without them has
    # the same tensors and must give the same bits
    prob = synth.prefill_problem(lens=[300, 0, 1, 129, 0], hq=32, hkv=8, block=128, seed=51)
    got = run_fused(prob)
    ref_out, ref_lse = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale)
    assert_forward_parity(*got, ref_out, ref_lse, "prefill with empty sequences")
    dense = synth.prefill_problem(lens=[300, 1, 129], hq=32, hkv=8, block=128, seed=51)
    np.testing.assert_array_equal(dense.q, prob.q)
    assert_bitwise(run_fused(dense), got, "empty sequences removed")
    assert_bitwise(run_states_merge(prob, cp=2, layout=1, rank_order=[1, 0]), got, "states + merge, CP 2")


def test_prefill_128_sequences():
    lens = synth.rng(52, synth.T_LENS).integers(1, 161, size=128).tolist()
    prob = synth.prefill_problem(lens=lens, hq=8, hkv=2, block=128, seed=52)
    got = run_fused(prob)
    ref_out, ref_lse = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale)
    assert_forward_parity(*got, ref_out, ref_lse, "128 sequences")
    order = list(np.random.default_rng(53).permutation(128))
    perm = synth.permute_batch(prob, order)
    moved = run_fused(perm)
    for new_s, old_s in enumerate(order):
        a, b = perm.cu_q[new_s], perm.cu_q[new_s + 1]
        c, d = prob.cu_q[old_s], prob.cu_q[old_s + 1]
        assert_bitwise(tuple(x[a:b] for x in moved), tuple(x[c:d] for x in got), f"sequence {old_s}")


def test_chunk_of_zero_queries():
    # sequence 0 has a 200-token cache and no new query; sequence 1 a chunk of
    # 100 queries over a 300-token cache
    prob = synth.prefill_problem(lens=[0, 100], kv_lens=[200, 300], hq=16, hkv=4, block=128, seed=54)
    got = run_fused(prob)
    ref_out, ref_lse = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale)
    assert_forward_parity(*got, ref_out, ref_lse, "chunk with an empty query range")


def test_decode_one_long_context():
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    dec = synth.paged_decode_problem(ctx=[131072], hq=32, hkv=8, seed=55, garbage_tail=False)
    qd = dv.bf16_to_device(dec.q)
    kp = torch.from_numpy(dec.k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(dec.v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ptd = dv.i32_to_device(dec.page_table)
    p = rlk.make_params(1, 32, 8, 128, softmax_scale=dec.scale)
    args = (p, qd, kp, vp, dec.k_bits.shape[0], dec.page_size, ptd, dec.page_table.shape[1], dec.seqlens)
    out, outb, lse = empty_outputs(torch, 1, 32)
    rlk.rlk_attn_decode_paged(*args, out, outb, lse)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, dec.seqlens), dtype=torch.uint8,
                     device="cuda")
    sout, soutb, slse = empty_outputs(torch, 1, 32)
    rlk.rlk_attn_decode_paged_splitk(*args, 0, sout, soutb, slse, ws)  # the library picks k
    rlk.rlk_attn_check_device_error()
    single = (out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy())
    split = (sout.cpu().numpy(), soutb.float().cpu().numpy(), slse.cpu().numpy())
    assert rlk.rlk_attn_decode_auto_split(p, dec.seqlens, torch.cuda.get_device_properties(0).multi_processor_count) > 1
    assert_bitwise(split, single, "split decode vs single pass")
    ref_out, ref_lse = oracle.decode_paged_f64(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seqlens, dec.scale)
    # out against the FP64 definition (the 2e-5 / one-ulp gates); the lse is
    # checked below, so the GPU's own lse stands in here
    assert_forward_parity(*single, ref_out, single[2], "decode over 131,072 tokens")
    # lse: 1023 sequential FP32 folds of a running lse near 12 (FP32 ulp
    # 9.5e-7 there) drift from the FP64 value by about sqrt(1023) half-ulps,
    # past the 1e-5 gate stated for the benchmark contexts (<= 256 blocks).
    # What the canonical fold fixes is checked instead: the GPU lse equals the
    # oracle's FP32 canonical fold of the exact block states to a few ulps (the
    # states' own FP32 rounding), and is no further from the FP64 value than
    # that fold is, plus those ulps
    ks, vs = dec.seq_kv(0)
    nb = (131072 + 127) // 128
    cu_q, cu_k = np.array([0, 1], np.int32), np.array([0, 131072], np.int32)
    worst_fold = 0.0
    for h in range(32):
        o_b, lse_b = oracle.row_block_states_f64(dec.q, ks, vs, cu_q, cu_k, dec.scale, 128, 0, h)
        assert len(lse_b) == nb
        _, l32 = oracle.fold_f32(np.arange(nb), o_b.astype(np.float32), lse_b.astype(np.float32))
        assert abs(float(single[2][0, h]) - l32) <= 4e-6, f"head {h}: GPU lse vs canonical FP32 fold"
        worst_fold = max(worst_fold, abs(l32 - float(ref_lse[0, h])))
    assert float(np.abs(single[2] - ref_lse).max()) <= worst_fold + 4e-6


def test_merge_rejects_slab_past_the_state_table():
    # a slab whose offset is valid in itself but whose rows reach past the
    # table (offset + Hq * row_count > n_state_pairs) must not be read: the
    # merge reports a bad state table, leaves that block missing, and the
    # context stays usable for the next call
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    from tests.gpu_helpers import device_inputs, params_of, to_np
    prob = synth.prefill_problem(lens=[300, 129], hq=32, hkv=8, block=128, seed=57)
    q, k, v = device_inputs(prob)
    p = params_of(prob)
    slabs, npairs = rlk.rlk_attn_plan_states(p, prob.cu_q, prob.cu_k, -1, 0)
    so = torch.empty((npairs, 128), dtype=torch.float32, device="cuda")
    sl = torch.empty((npairs,), dtype=torch.float32, device="cuda")
    rlk.rlk_attn_prefill_states(p, q, k, v, prob.cu_q, prob.cu_k, -1, 0, so, sl)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, prob.cu_q, prob.cu_k), dtype=torch.uint8,
                     device="cuda")
    bad = slabs.copy()
    last = int(np.argmax(bad["offset"]))
    bad["offset"][last] = npairs - prob.hq * int(bad["row_count"][last]) + 1  # one pair past the end
    out, outb, lse = empty_outputs(torch, q.shape[0], prob.hq)
    rlk.rlk_attn_merge_states(p, prob.cu_q, prob.cu_k, dv.slabs_to_device(bad), len(bad), so, sl, out, outb, lse, ws)
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_check_device_error()
    assert e.value.status == 9  # RLK_ERR_BAD_STATE_TABLE
    # the rows needing that block are NaN (missing), the others are merged
    got = to_np(out, outb, lse)
    assert np.isnan(got[2]).any() and not np.isnan(got[2]).all()
    # the same table with the right offset merges cleanly afterwards
    good = empty_outputs(torch, q.shape[0], prob.hq)
    rlk.rlk_attn_merge_states(p, prob.cu_q, prob.cu_k, dv.slabs_to_device(slabs), len(slabs), so, sl, *good, ws)
    rlk.rlk_attn_check_device_error()
    assert_bitwise(to_np(*good), run_fused(prob), "merge after a rejected table")
