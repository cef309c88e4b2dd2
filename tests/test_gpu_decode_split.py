"""Split decode (rlk_attn_decode_paged_splitk): each sequence's KV blocks in
split_k fixed ranges processed by different SMs, block states written out
and folded in ascending global_block_index order -- bit for bit the
single-pass decode whatever split_k, and within the tolerances of the oracle
("[WS2][Attention] H100 validation and reproduction guide", Status: fixed
global_block_index merge, decode/prefill max abs 0.0)."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import assert_bitwise, assert_forward_parity, empty_outputs, lib, torch_cuda
from tests.test_gpu_decode import run_decode

pytestmark = pytest.mark.gpu


def run_split(dec, split_k):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    q = dv.bf16_to_device(dec.q)
    kp = torch.from_numpy(dec.k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(dec.v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ptd = dv.i32_to_device(dec.page_table)
    n = len(dec.seqlens)
    out, outb, lse = empty_outputs(torch, n, dec.hq)
    p = rlk.make_params(n, dec.hq, dec.hkv, 128, softmax_scale=dec.scale)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, dec.seqlens), dtype=torch.uint8,
                     device="cuda")
    rlk.rlk_attn_decode_paged_splitk(p, q, kp, vp, dec.k_bits.shape[0], dec.page_size, ptd, dec.page_table.shape[1],
                                     dec.seqlens, split_k, out, outb, lse, ws)
    rlk.rlk_attn_check_device_error()
    return out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy()


@pytest.fixture(scope="module")
def dec():
    return synth.paged_decode_problem(ctx=[1, 17, 128, 129, 1000, 2049, 4096], seed=51, spare_pages=4)


@pytest.mark.parametrize("split_k", [0, 1, 2, 3, 8, 64])  # 0: the library picks k
def test_split_decode_equals_single_pass(dec, split_k):
    assert_bitwise(run_split(dec, split_k), run_decode(dec), f"split_k {split_k}")


def test_split_decode_parity(dec):
    out, outb, lse = run_split(dec, 4)
    ref_out, ref_lse = oracle.decode_paged_f64(dec.q, dec.k_pool, dec.v_pool, dec.page_table, dec.seqlens, dec.scale)
    assert_forward_parity(out, outb, lse, ref_out, ref_lse, "split decode")


@pytest.mark.parametrize("hq,hkv", [(8, 8), (32, 4)])
def test_split_decode_group_sizes(hq, hkv):
    d = synth.paged_decode_problem(ctx=[5, 300, 1500], hq=hq, hkv=hkv, seed=52)
    assert_bitwise(run_split(d, 5), run_decode(d), f"hq{hq}/hkv{hkv}")


def test_split_decode_fold_on_chip_long():
    # 4 x 32768 tokens (the long-context split workload): 32 (sequence, KV
    # head) pairs, so k = 4 and the library's own choice run as one
    # cooperative launch with the fold on chip, k = 8 as contiguous ranges
    # and the fold kernel; every call, repeated, equals the single pass bit
    # for bit
    d = synth.paged_decode_problem(ctx=[32768] * 4, seed=53)
    ref = run_decode(d)
    for k in (4, 0, 4, 8):
        assert_bitwise(run_split(d, k), ref, f"4 x 32768, split_k {k}")


@pytest.mark.parametrize("hq,hkv,k", [(24, 8, 3), (40, 8, 2), (8, 8, 7)])
def test_split_decode_fold_on_chip_group_shapes(hq, hkv, k):
    # the on-chip fold with groups of 3, 5 and 1 query heads per KV head,
    # partial last blocks and a one-block sequence (fewer items than k)
    d = synth.paged_decode_problem(ctx=[1, 200, 1999, 4097], hq=hq, hkv=hkv, seed=54)
    assert_bitwise(run_split(d, k), run_decode(d), f"hq{hq}/hkv{hkv} k {k}")
