"""GPU parity of RoPE: the streaming pass (one tensor, or queries and keys in
one launch) equals the oracle's canonical FP32 RoPE bit for bit (BF16
results are byte-exact work); the prefill's and the decode kernel's
in-kernel query RoPE equal the pass followed by the plain kernel, which in
turn matches the oracle (prefill) and the last row of the prefill over
rotated inputs (decode) ("WS2 Attention PR5
Drift Benchmark", Scope: RoPE composed before Attention, Attention consuming
post-RoPE Q/K; "[WS2][Attention] H100 validation and reproduction guide", PR
stack: decode KV-cache replay and cache/position/RoPE identity)."""
import numpy as np
import pytest

import oracle
from deterministic_context_attention_gb300 import synth
from tests.gpu_helpers import assert_bitwise, assert_forward_parity, empty_outputs, lib, run_fused, torch_cuda

pytestmark = pytest.mark.gpu

THETA = 1.0e6


def table_dev(max_pos):
    torch = torch_cuda()
    return torch.from_numpy(lib().rlk_attn_rope_table(THETA, max_pos)).cuda()


def gpu_rope(x, cu, pos_offset, max_pos, inplace=False):
    """x [T, H, 128] BF16 values (float32) through rlk_attn_rope."""
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    xd = dv.bf16_to_device(x)
    yd = xd if inplace else torch.full_like(xd, float("nan"))
    p = rlk.make_params(len(cu) - 1)
    rlk.rlk_attn_rope(p, xd, yd, x.shape[1], cu, pos_offset, table_dev(max_pos), max_pos)
    rlk.rlk_attn_check_device_error()
    return yd.float().cpu().numpy()


def positions(cu, pos_offset):
    return np.concatenate([np.arange(cu[s + 1] - cu[s], dtype=np.int64) + (0 if pos_offset is None else pos_offset[s])
                           for s in range(len(cu) - 1)]).astype(np.int32)


@pytest.mark.parametrize("heads,inplace", [(32, False), (8, True), (3, False)])
def test_rope_pass_equals_oracle_bitwise(heads, inplace):
    # ragged lengths with an empty sequence, offsets from 0 to 40,000
    lens = [300, 0, 129, 1, 1000]
    offs = np.array([0, 7, 100, 40000, 3], np.int32)
    cu = synth.cu_seqlens(lens)
    x = synth.normal_bf16(41, synth.T_Q, (int(cu[-1]), heads, 128))
    y = gpu_rope(x, cu, offs, 41001, inplace)
    ref = oracle.rope_f32(x, positions(cu, offs), THETA)
    np.testing.assert_array_equal(y, ref)


def test_rope_pass_prefill_workload_bitwise():
    # the query tensor of the varlen prefill workload, positions 0..len-1
    cfg = synth.CFG_PREFILL
    cu = synth.cu_seqlens(cfg["lens"])
    x = synth.normal_bf16(cfg["seed"], synth.T_Q, (int(cu[-1]), cfg["hq"], 128))
    y = gpu_rope(x, cu, None, 4096)
    np.testing.assert_array_equal(y, oracle.rope_f32(x, positions(cu, None), THETA))


def test_rope_chunked_positions_equal_full_rows():
    # a chunk of q_len rows at offset kv_len - q_len gives the full rows' bits
    cu_full = synth.cu_seqlens([700])
    x = synth.normal_bf16(43, synth.T_K, (700, 8, 128))
    full = gpu_rope(x, cu_full, None, 700)
    chunk = gpu_rope(x[500:], synth.cu_seqlens([200]), np.array([500], np.int32), 700)
    assert_bitwise((chunk,), (full[500:],), "chunk rows")


def run_decode_q(dec, q, rope_max_pos=None):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    qd = dv.bf16_to_device(q)
    kp = torch.from_numpy(dec.k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(dec.v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    ptd = dv.i32_to_device(dec.page_table)
    n = len(dec.seqlens)
    out, outb, lse = empty_outputs(torch, n, dec.hq)
    p = rlk.make_params(n, dec.hq, dec.hkv, 128, softmax_scale=dec.scale)
    if rope_max_pos is None:
        rlk.rlk_attn_decode_paged(p, qd, kp, vp, dec.k_bits.shape[0], dec.page_size, ptd, dec.page_table.shape[1],
                                  dec.seqlens, out, outb, lse)
    else:
        rlk.rlk_attn_decode_paged_rope(p, qd, kp, vp, dec.k_bits.shape[0], dec.page_size, ptd,
                                       dec.page_table.shape[1], dec.seqlens, table_dev(rope_max_pos), rope_max_pos,
                                       out, outb, lse)
    rlk.rlk_attn_check_device_error()
    return out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("hq,hkv", [(32, 8), (8, 8), (32, 4), (24, 8)])
def test_decode_rope_equals_pass_then_decode(hq, hkv):
    dec = synth.paged_decode_problem(ctx=[1, 17, 128, 129, 1000, 2049], hq=hq, hkv=hkv, seed=44, spare_pages=3)
    n = len(dec.seqlens)
    fused = run_decode_q(dec, dec.q, rope_max_pos=4096)
    q_rot = gpu_rope(dec.q, np.arange(n + 1, dtype=np.int32), dec.seqlens - 1, 4096)
    plain = run_decode_q(dec, q_rot)
    assert_bitwise(fused, plain, "in-kernel RoPE vs pass + decode")
    q_ref = oracle.rope_f32(dec.q, dec.seqlens - 1, THETA)
    ref_out, ref_lse = oracle.decode_paged_f64(q_ref, dec.k_pool, dec.v_pool, dec.page_table, dec.seqlens, dec.scale)
    assert_forward_parity(*fused, ref_out, ref_lse, "decode with RoPE")


@pytest.mark.parametrize("split_k", [0, 3])
def test_split_decode_rope_equals_single_pass(split_k):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    dec = synth.paged_decode_problem(ctx=[1, 129, 1000, 3000], hq=32, hkv=8, seed=47, spare_pages=2)
    n = len(dec.seqlens)
    single = run_decode_q(dec, dec.q, rope_max_pos=4096)
    qd = dv.bf16_to_device(dec.q)
    kp = torch.from_numpy(dec.k_bits.view(np.int16)).cuda().view(torch.bfloat16)
    vp = torch.from_numpy(dec.v_bits.view(np.int16)).cuda().view(torch.bfloat16)
    p = rlk.make_params(n, dec.hq, dec.hkv, 128, softmax_scale=dec.scale)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, dec.seqlens), dtype=torch.uint8,
                     device="cuda")
    out, outb, lse = empty_outputs(torch, n, dec.hq)
    rlk.rlk_attn_decode_paged_splitk_rope(p, qd, kp, vp, dec.k_bits.shape[0], dec.page_size,
                                          dv.i32_to_device(dec.page_table), dec.page_table.shape[1], dec.seqlens,
                                          split_k, table_dev(4096), 4096, out, outb, lse, ws)
    rlk.rlk_attn_check_device_error()
    assert_bitwise((out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy()), single,
                   f"split {split_k} with RoPE")


def test_rope_cache_position_identity():
    # prefill over RoPE'd q and k; decode of the last token (pre-RoPE query,
    # cache filled with the RoPE'd keys through a permuted page table) gives
    # the prefill's last row bit for bit
    torch = torch_cuda()
    hq, hkv, ctx, ps = 32, 8, 1000, 16
    q = synth.normal_bf16(45, synth.T_Q, (ctx, hq, 128))
    k = synth.normal_bf16(45, synth.T_K, (ctx, hkv, 128))
    v = synth.normal_bf16(45, synth.T_V, (ctx, hkv, 128))
    cu = np.array([0, ctx], np.int32)
    q_rot = gpu_rope(q, cu, None, ctx)
    k_rot = gpu_rope(k, cu, None, ctx)
    prob = synth.Prefill(q_rot, k_rot, v, cu, cu, hq, hkv, 128, 1.0 / np.sqrt(128), 128)
    po, pb, pl = run_fused(prob)
    npg = (ctx + ps - 1) // ps
    perm = np.random.default_rng(46).permutation(npg).astype(np.int32)
    kb = np.zeros((npg, ps, hkv, 128), np.uint16)
    vb = np.zeros((npg, ps, hkv, 128), np.uint16)
    pad = npg * ps - ctx
    kb[perm] = np.concatenate([synth.bf16_bits(k_rot), np.zeros((pad, hkv, 128), np.uint16)]).reshape(npg, ps, hkv, 128)
    vb[perm] = np.concatenate([synth.bf16_bits(v), np.zeros((pad, hkv, 128), np.uint16)]).reshape(npg, ps, hkv, 128)
    dec = synth.PagedDecode(q[-1:], kb, vb, perm[None, :], np.array([ctx], np.int32), ps, hq, hkv, 128,
                            1.0 / np.sqrt(128), 46)
    d = run_decode_q(dec, q[-1:], rope_max_pos=ctx)
    assert_bitwise(d, (po[-1:], pb[-1:], pl[-1:]), "decode with RoPE vs prefill last row")


def _prefill_rope(prob, q_raw, k_rot, cp=1, ranks=None):
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    from tests.gpu_helpers import params_of, to_np
    qd, kd, vd = dv.bf16_to_device(q_raw), dv.bf16_to_device(k_rot), dv.bf16_to_device(prob.v)
    max_pos = int(np.diff(prob.cu_k).max())
    out, outb, lse = empty_outputs(torch, qd.shape[0], prob.hq)
    p = params_of(prob, cp, 1)
    for r in (ranks if ranks is not None else [-1]):
        rlk.rlk_attn_prefill_rope(p, qd, kd, vd, prob.cu_q, prob.cu_k, r, table_dev(max_pos), max_pos, out, outb, lse)
    rlk.rlk_attn_check_device_error()
    return to_np(out, outb, lse)


@pytest.mark.parametrize("lens,kv_extra,block", [([4096, 3000, 1024, 777], 0, 128), ([300, 1, 129], 37, 64)])
def test_prefill_with_in_kernel_rope(lens, kv_extra, block):
    # pre-RoPE queries rotated inside the prefill kernel at positions
    # kv_len - q_len + i, post-RoPE keys: bit-identical to the RoPE pass on
    # the queries followed by the plain prefill, and within the gates of the
    # oracle's attention over the oracle-rotated queries.  The second case is
    # a chunk of queries over a longer KV cache (positions offset by 37).
    kv = [n + kv_extra for n in lens]
    prob = synth.prefill_problem(lens=lens, hq=32, hkv=8, block=block, seed=81, kv_lens=kv)
    q_raw = synth.normal_bf16(82, synth.T_Q, prob.q.shape)
    k_rot = oracle.rope_f32(prob.k, positions(prob.cu_k, None), THETA)
    offs = (np.diff(prob.cu_k) - np.diff(prob.cu_q)).astype(np.int32)
    max_pos = int(np.diff(prob.cu_k).max())
    q_rot = gpu_rope(q_raw, prob.cu_q, offs, max_pos)
    np.testing.assert_array_equal(q_rot, oracle.rope_f32(q_raw, positions(prob.cu_q, offs), THETA))
    rotated = synth.Prefill(q_rot, k_rot, prob.v, prob.cu_q, prob.cu_k, prob.hq, prob.hkv, prob.d, prob.scale,
                            prob.block)
    fused = _prefill_rope(prob, q_raw, k_rot)
    assert_bitwise(fused, run_fused(rotated), "in-kernel RoPE vs pass + prefill")
    assert_bitwise(_prefill_rope(prob, q_raw, k_rot, cp=2, ranks=[1, 0]), fused, "in-kernel RoPE, CP 2")
    rows = np.sort(np.random.default_rng(83).choice(int(prob.cu_q[-1]), 120, replace=False))
    ref_out, ref_lse = oracle.attention_f64(q_rot, k_rot, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=rows)
    assert_forward_parity(*(x[rows] for x in fused), ref_out, ref_lse, "prefill with in-kernel RoPE")


@pytest.mark.parametrize("keep", ["f32", "bf16"])
def test_prefill_rope_single_output(keep):
    # whole sequences rotate their queries through the output buffer they
    # are given: with only the FP32 or only the BF16 output, the result is
    # the two-output call's, bit for bit
    lens = [700, 129, 1]
    prob = synth.prefill_problem(lens=lens, hq=32, hkv=8, block=128, seed=84, kv_lens=[n + 5 for n in lens])
    q_raw = synth.normal_bf16(85, synth.T_Q, prob.q.shape)
    k_rot = oracle.rope_f32(prob.k, positions(prob.cu_k, None), THETA)
    ref_out, ref_outb, ref_lse = _prefill_rope(prob, q_raw, k_rot)
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    from tests.gpu_helpers import params_of
    qd, kd, vd = dv.bf16_to_device(q_raw), dv.bf16_to_device(k_rot), dv.bf16_to_device(prob.v)
    max_pos = int(np.diff(prob.cu_k).max())
    out, outb, lse = empty_outputs(torch, qd.shape[0], prob.hq)
    rlk.rlk_attn_prefill_rope(params_of(prob, 1, 1), qd, kd, vd, prob.cu_q, prob.cu_k, -1, table_dev(max_pos), max_pos,
                              out if keep == "f32" else None, outb if keep == "bf16" else None, lse)
    rlk.rlk_attn_check_device_error()
    np.testing.assert_array_equal(lse.cpu().numpy(), ref_lse)
    if keep == "f32":
        np.testing.assert_array_equal(out.cpu().numpy(), ref_out)
    else:
        np.testing.assert_array_equal(outb.float().cpu().numpy(), ref_outb)
    # the queries themselves are not modified
    np.testing.assert_array_equal(qd.cpu().view(torch.int16).numpy().view(np.uint16), synth.bf16_bits(q_raw))


def test_rope_qk_single_launch_equals_two_passes():
    # queries and keys of the same tokens in one launch, bit for bit the two
    # single-tensor passes (ragged lengths, an empty sequence, offsets)
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    lens = [300, 0, 129, 1, 1000]
    offs = np.array([0, 7, 100, 4000, 3], np.int32)
    cu = synth.cu_seqlens(lens)
    q = dv.bf16_to_device(synth.normal_bf16(91, synth.T_Q, (int(cu[-1]), 32, 128)))
    k = dv.bf16_to_device(synth.normal_bf16(91, synth.T_K, (int(cu[-1]), 8, 128)))
    table = table_dev(5001)
    p = rlk.make_params(len(lens), 32, 8)
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    rlk.rlk_attn_rope_qk(p, q, qo, k, ko, cu, offs, table, 5001)
    q1, k1 = torch.empty_like(q), torch.empty_like(k)
    rlk.rlk_attn_rope(p, q, q1, 32, cu, offs, table, 5001)
    rlk.rlk_attn_rope(p, k, k1, 8, cu, offs, table, 5001)
    rlk.rlk_attn_check_device_error()
    assert torch.equal(qo.view(torch.int16), q1.view(torch.int16))
    assert torch.equal(ko.view(torch.int16), k1.view(torch.int16))


def test_prefill_rope_graph_replay():
    # the RoPE pass into the output buffer and the prefill after it, captured
    # in one CUDA graph: replays with new queries copied in equal the eager
    # call on those queries bit for bit
    torch = torch_cuda()
    rlk = lib()
    from deterministic_context_attention_gb300 import device as dv
    from tests.gpu_helpers import params_of
    lens = [1000, 300, 129]
    prob = synth.prefill_problem(lens=lens, hq=32, hkv=8, block=128, seed=86, kv_lens=[n + 3 for n in lens])
    k_rot = oracle.rope_f32(prob.k, positions(prob.cu_k, None), THETA)
    qs = [synth.normal_bf16(87 + i, synth.T_Q, prob.q.shape) for i in range(2)]
    refs = [_prefill_rope(prob, q_raw, k_rot) for q_raw in qs]
    max_pos = int(np.diff(prob.cu_k).max())
    table = table_dev(max_pos)
    qd, kd, vd = dv.bf16_to_device(qs[0]), dv.bf16_to_device(k_rot), dv.bf16_to_device(prob.v)
    out, outb, lse = empty_outputs(torch, qd.shape[0], prob.hq)
    p = params_of(prob, 1, 1)

    def call():
        rlk.rlk_attn_prefill_rope(p, qd, kd, vd, prob.cu_q, prob.cu_k, -1, table, max_pos, out, outb, lse)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    for i in (1, 0, 1):
        qd.copy_(dv.bf16_to_device(qs[i]))
        graph.replay()
        torch.cuda.synchronize()
        rlk.rlk_attn_check_device_error()
        assert_bitwise((out.cpu().numpy(), outb.float().cpu().numpy(), lse.cpu().numpy()), refs[i],
                       f"graph replay with queries {i}")
