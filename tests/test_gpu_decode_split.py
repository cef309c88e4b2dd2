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


def _split_inputs(torch, dv, d):
    q = dv.bf16_to_device(d.q)
    kp = torch.from_numpy(d.k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(d.v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    return q, kp, vp, dv.i32_to_device(d.page_table)


def test_split_decode_fold_on_chip_reused_workspace():
    # the on-chip fold's items fill their own table slots and publish a flag
    # per call: one workspace, pre-filled with values that look like landed
    # states (zeros) and then reused across calls with other inputs, never
    # lets a fold read an earlier call's states
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    probs = [synth.paged_decode_problem(ctx=[4097, 2000, 300, 128], seed=s) for s in (55, 56)]
    refs = [run_decode(d) for d in probs]
    d0 = probs[0]
    p = rlk.make_params(4, d0.hq, d0.hkv, 128, softmax_scale=d0.scale)
    ws = torch.zeros(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, d0.seqlens), dtype=torch.uint8,
                     device="cuda")
    for i in (0, 1, 0, 1, 1):
        d = probs[i]
        q, kp, vp, ptd = _split_inputs(torch, dv, d)
        out, outb, lse = empty_outputs(torch, 4, d.hq)
        rlk.rlk_attn_decode_paged_splitk(p, q, kp, vp, d.k_bits.shape[0], d.page_size, ptd, d.page_table.shape[1],
                                         d.seqlens, 4, out, outb, lse, ws)
        rlk.rlk_attn_check_device_error()
        got = (out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy())
        assert_bitwise(got, refs[i], f"call with inputs {i}")


def test_split_decode_fold_on_chip_graph_replay():
    # inside a CUDA graph the call fills the table before the launch (a
    # replay reuses the launch's arguments, flags included): replays with new
    # inputs copied in equal the single pass on those inputs
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    probs = [synth.paged_decode_problem(ctx=[4097, 2000, 300, 128], seed=s) for s in (57, 58)]
    refs = [run_decode(d) for d in probs]
    d0 = probs[0]
    p = rlk.make_params(4, d0.hq, d0.hkv, 128, softmax_scale=d0.scale)
    bufs = _split_inputs(torch, dv, d0)
    q, kp, vp, ptd = (b.clone() for b in bufs)
    out, outb, lse = empty_outputs(torch, 4, d0.hq)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, d0.seqlens), dtype=torch.uint8,
                     device="cuda")

    def call():
        rlk.rlk_attn_decode_paged_splitk(p, q, kp, vp, d0.k_bits.shape[0], d0.page_size, ptd,
                                         d0.page_table.shape[1], d0.seqlens, 4, out, outb, lse, ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()  # configures the kernels outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for i in (1, 0, 1):
        d = probs[i]
        assert d.k_bits.shape == d0.k_bits.shape and d.page_table.shape == d0.page_table.shape
        for dst, src in zip((q, kp, vp, ptd), _split_inputs(torch, dv, d)):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        rlk.rlk_attn_check_device_error()
        got = (out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy())
        assert_bitwise(got, refs[i], f"graph replay with inputs {i}")
