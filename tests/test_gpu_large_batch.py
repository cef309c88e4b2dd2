"""Batches of more than 128 sequences (one launch's sequence tables hold
128; a larger call runs as consecutive 128-sequence ranges): every entry
point gives, bit for bit, what calls on 128-sequence subsets give, and
matches the oracle on sampled sequences ("[WS2][Cross-config][Attention]
Integrate the Qwen3-8B TP=2 CP=2 BF16 Attention setting", the contract knobs:
batch invariance belongs to identity; "[WS2][Attention] H100 validation and
reproduction guide", Status: strict decode/prefill max abs 0.0)."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import (assert_bitwise, assert_forward_parity, device_inputs, empty_outputs, lib,
                               params_of, run_fused, run_states_merge, to_np, torch_cuda)

pytestmark = pytest.mark.gpu


def _decode(dec, seqs, split_k=None):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    q = dv.bf16_to_device(dec.q[seqs])
    kp = torch.from_numpy(dec.k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(dec.v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    pt = dec.page_table[seqs]
    ptd = dv.i32_to_device(pt)
    ctx = dec.seqlens[seqs]
    out, outb, lse = empty_outputs(torch, len(seqs), dec.hq)
    p = rlk.make_params(len(seqs), dec.hq, dec.hkv, 128, softmax_scale=dec.scale)
    if split_k is None:
        rlk.rlk_attn_decode_paged(p, q, kp, vp, dec.k_bits.shape[0], dec.page_size, ptd, pt.shape[1], ctx, out, outb,
                                  lse)
    else:
        ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, ctx), dtype=torch.uint8,
                         device="cuda")
        rlk.rlk_attn_decode_paged_splitk(p, q, kp, vp, dec.k_bits.shape[0], dec.page_size, ptd, pt.shape[1], ctx,
                                         split_k, out, outb, lse, ws)
    rlk.rlk_attn_check_device_error()
    return to_np(out, outb, lse)


@pytest.fixture(scope="module")
def dec512():
    return synth.paged_decode_problem(n=512, ctx_lo=1, ctx_hi=400, hq=8, hkv=2, seed=71)


def test_decode_512_sequences(dec512):
    dec = dec512
    allseq = np.arange(512)
    full = _decode(dec, allseq)
    for s0 in range(0, 512, 128):
        part = _decode(dec, allseq[s0:s0 + 128])
        assert_bitwise(part, tuple(a[s0:s0 + 128] for a in full), f"sequences {s0}..{s0 + 127}")
    pick = np.sort(np.random.default_rng(72).choice(512, 150, replace=False))
    assert_bitwise(_decode(dec, pick), tuple(a[pick] for a in full), "150 scattered sequences")
    sample = pick[:40]
    ref_out, ref_lse = oracle.decode_paged_f64(dec.q[sample], dec.k_pool, dec.v_pool, dec.page_table[sample],
                                               dec.seqlens[sample], dec.scale)
    assert_forward_parity(*(a[sample] for a in full), ref_out, ref_lse, "512-sequence decode")
    for k in (0, 3):
        assert_bitwise(_decode(dec, allseq, split_k=k), full, f"split decode k={k}")


@pytest.fixture(scope="module")
def pre300():
    lens = synth.rng(73, synth.T_LENS).integers(1, 161, size=300).tolist()
    return synth.prefill_problem(lens=lens, hq=8, hkv=2, block=128, seed=73)


def _subset(prob, seqs):
    """The prefill problem of a contiguous sequence range."""
    a, b = int(prob.cu_q[seqs[0]]), int(prob.cu_q[seqs[-1] + 1])
    c, d = int(prob.cu_k[seqs[0]]), int(prob.cu_k[seqs[-1] + 1])
    return synth.Prefill(prob.q[a:b], prob.k[c:d], prob.v[c:d], prob.cu_q[seqs[0]:seqs[-1] + 2] - a,
                         prob.cu_k[seqs[0]:seqs[-1] + 2] - c, prob.hq, prob.hkv, prob.d, prob.scale, prob.block)


def test_prefill_300_sequences(pre300):
    prob = pre300
    full = run_fused(prob)
    for s0 in range(0, 300, 128):
        seqs = list(range(s0, min(300, s0 + 128)))
        a, b = int(prob.cu_q[seqs[0]]), int(prob.cu_q[seqs[-1] + 1])
        assert_bitwise(run_fused(_subset(prob, seqs)), tuple(x[a:b] for x in full), f"sequences {s0}..")
    assert_bitwise(run_states_merge(prob, cp=2, layout=1, rank_order=[1, 0], shuffle_seed=5), full,
                   "states + merge, CP 2, 300 sequences")
    assert_bitwise(run_fused(prob, cp=4, layout=0, ranks=[3, 1, 0, 2]), full, "fused CP 4, 300 sequences")
    rows = np.sort(np.random.default_rng(74).choice(int(prob.cu_q[-1]), 200, replace=False))
    ref_out, ref_lse = oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=rows)
    assert_forward_parity(*(x[rows] for x in full), ref_out, ref_lse, "300-sequence prefill")


def test_rope_and_backward_300_sequences(pre300):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    prob = pre300
    q, k, v = device_inputs(prob)
    max_pos = int(np.diff(prob.cu_q).max())
    table = torch.from_numpy(rlk.rlk_attn_rope_table(1.0e6, max_pos)).cuda()
    pr = rlk.make_params(300)
    rot = torch.empty_like(q)
    rlk.rlk_attn_rope(pr, q, rot, prob.hq, prob.cu_q, None, table, max_pos)
    for s0 in range(0, 300, 128):
        s1 = min(300, s0 + 128)
        a, b = int(prob.cu_q[s0]), int(prob.cu_q[s1])
        part = torch.empty_like(q[a:b])
        rlk.rlk_attn_rope(rlk.make_params(s1 - s0), q[a:b], part, prob.hq, prob.cu_q[s0:s1 + 1] - a, None, table,
                          max_pos)
        assert torch.equal(part.view(torch.int16), rot[a:b].view(torch.int16)), f"RoPE sequences {s0}.."
    rlk.rlk_attn_check_device_error()
    # backward over the whole batch against the ranges, and against the oracle
    from tests.test_gpu_backward import assert_grad_parity, forward_and_backward
    dout = synth.normal_bf16(75, synth.T_DOUT, prob.q.shape)
    dq, dk, dvv = forward_and_backward(prob, dout, qkv=(q, k, v))
    seqs = list(range(128, 256))
    sub = _subset(prob, seqs)
    a, b = int(prob.cu_q[128]), int(prob.cu_q[256])
    sq, sk, sv = forward_and_backward(sub, dout[a:b])
    for x, y, name in ((sq, dq[a:b], "dq"), (sk, dk[a:b], "dk"), (sv, dvv[a:b], "dv")):
        assert np.array_equal(x.view(np.uint32), y.view(np.uint32)), f"backward {name}, sequences 128..255"
    rq, rk, rv = oracle.backward_f64(prob.q, prob.k, prob.v, dout, prob.cu_q, prob.scale)
    for got, ref, name in ((dq, rq, "dq"), (dk, rk, "dk"), (dvv, rv, "dv")):
        assert_grad_parity(got, ref, f"300-sequence {name}")
