"""GPU parity and invariance of paged-KV decode: against the oracle, equal
bit for bit to the last row of the equivalent full prefill, invariant to page
permutation and batch subset ("[WS2][Attention] H100 validation and
reproduction guide", PR stack: decode KV-cache replay, paged-KV adapter;
Status: strict decode/prefill Out/LSE max abs 0.0)."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import assert_bitwise, assert_forward_parity, empty_outputs, lib, run_fused, torch_cuda

pytestmark = pytest.mark.gpu


def run_decode(dec, page_table=None, k_bits=None, v_bits=None, seqs=None, block=128):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    seqs = list(range(len(dec.seqlens))) if seqs is None else list(seqs)
    pt = dec.page_table if page_table is None else page_table
    kb = dec.k_bits if k_bits is None else k_bits
    vb = dec.v_bits if v_bits is None else v_bits
    q = dv.bf16_to_device(dec.q[seqs])
    kp = torch.from_numpy(kb.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(vb.view(np.int16)).cuda().view(torch.bfloat16)
    ptd = dv.i32_to_device(pt[seqs])
    out, outb, lse = empty_outputs(torch, len(seqs), dec.hq)
    p = rlk.make_params(len(seqs), dec.hq, dec.hkv, block, softmax_scale=dec.scale)
    rlk.rlk_attn_decode_paged(p, q, kp, vp, kb.shape[0], dec.page_size, ptd, pt.shape[1], dec.seqlens[seqs],
                              out, outb, lse)
    rlk.rlk_attn_check_device_error()
    return out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy()


@pytest.fixture(scope="module")
def small_dec():
    # ragged contexts: 1 token, a partial page, exact pages, exact blocks, tails
    return synth.paged_decode_problem(ctx=[1, 15, 16, 17, 127, 128, 129, 300, 1000, 2049], seed=31,
                                      spare_pages=5)


def test_decode_parity(small_dec):
    out, outb, lse = run_decode(small_dec)
    ref_out, ref_lse = oracle.decode_paged_f64(small_dec.q, small_dec.k_pool, small_dec.v_pool,
                                               small_dec.page_table, small_dec.seqlens, small_dec.scale)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, "decode")


def test_decode_equals_last_prefill_row_bitwise(small_dec):
    out, outb, lse = run_decode(small_dec)
    for s in range(len(small_dec.seqlens)):
        ctx = int(small_dec.seqlens[s])
        ks, vs = small_dec.seq_kv(s)
        q = np.zeros((ctx, small_dec.hq, 128), np.float32)
        q[-1] = small_dec.q[s]
        cu = np.array([0, ctx], np.int32)
        prob = synth.Prefill(q, ks, vs, cu, cu, small_dec.hq, small_dec.hkv, 128, small_dec.scale, 128)
        po, pb, pl = run_fused(prob)
        assert_bitwise((out[s], outb[s], lse[s]), (po[-1], pb[-1], pl[-1]), f"sequence {s} (ctx {ctx})")
        # and the chunked form: one query over the whole cache
        one = synth.Prefill(q[-1:], ks, vs, np.array([0, 1], np.int32), cu, small_dec.hq, small_dec.hkv, 128,
                            small_dec.scale, 128)
        co, cb, cl = run_fused(one)
        assert_bitwise((out[s], outb[s], lse[s]), (co[0], cb[0], cl[0]), f"sequence {s} chunk-1 prefill")


def test_decode_page_permutation_and_subset(small_dec):
    base = run_decode(small_dec)
    n_pages = small_dec.k_bits.shape[0]
    perm = np.random.default_rng(4).permutation(n_pages)
    inv = np.argsort(perm)
    pt = np.where(small_dec.page_table >= 0, inv[np.maximum(small_dec.page_table, 0)], -1).astype(np.int32)
    moved = run_decode(small_dec, page_table=pt, k_bits=small_dec.k_bits[perm], v_bits=small_dec.v_bits[perm])
    assert_bitwise(moved, base, "page permutation")
    subset = [8, 2, 5]
    sub = run_decode(small_dec, seqs=subset)
    assert_bitwise(sub, tuple(x[subset] for x in base), "batch subset")


def test_bad_page_id_reported(small_dec):
    torch = torch_cuda()
    rlk = lib()
    pt = small_dec.page_table.copy()
    pt[3, 0] = 10 ** 6
    with pytest.raises(rlk.RlkError) as e:
        run_decode(small_dec, page_table=pt)
    assert e.value.status == 8  # RLK_ERR_BAD_PAGE
    rlk.rlk_attn_check_device_error()  # cleared
    del torch


# Query heads per KV head 1, 2, 4 and 8 run the transposed decode kernel (keys
# on the MMA's M side, one instantiation per padded group size); 16 heads per
# KV head and 64-key blocks run the forward engine's decode mode.  Every one
# matches the oracle and equals the last row of the same prefill bit for bit.
@pytest.mark.parametrize("hq,hkv,block", [(8, 8, 128), (16, 8, 128), (24, 8, 128), (32, 4, 128), (32, 2, 128),
                                          (32, 8, 64)])
def test_decode_group_sizes_and_block(hq, hkv, block):
    dec = synth.paged_decode_problem(ctx=[1, 64, 129, 300, 777], hq=hq, hkv=hkv, seed=41, spare_pages=3)
    out, outb, lse = run_decode(dec, block=block)
    ref_out, ref_lse = oracle.decode_paged_f64(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seqlens, dec.scale)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, f"decode hq{hq}/hkv{hkv} block {block}")
    for s in range(len(dec.seqlens)):
        ctx = int(dec.seqlens[s])
        ks, vs = dec.seq_kv(s)
        q = np.zeros((ctx, dec.hq, 128), np.float32)
        q[-1] = dec.q[s]
        cu = np.array([0, ctx], np.int32)
        prob = synth.Prefill(q, ks, vs, cu, cu, dec.hq, dec.hkv, 128, dec.scale, block)
        po, pb, pl = run_fused(prob)
        assert_bitwise((out[s], outb[s], lse[s]), (po[-1], pb[-1], pl[-1]), f"sequence {s} (ctx {ctx})")
