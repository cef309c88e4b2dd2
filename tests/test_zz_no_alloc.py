"""The workspace-free merge entry point, for callers that cannot allocate
device memory (graph capture, fixed-pool allocators, APIs that only pass
input and output buffers).

It must give the same result as rlk_attn_merge_states on the same state
table, on two calls in a row (the shared scratch keeps the previous call's
contents, which the entry point re-initialises).  This file is collected
last so that a run stopping at its first failure has run every other test.
"""
import numpy as np
import pytest

from deterministic_context_attention_gb300 import synth

pytestmark = pytest.mark.gpu


def _tables(prob, cp, rank_order, shuffle_seed):
    import torch
    import deterministic_context_attention_gb300 as rlk
    from deterministic_context_attention_gb300 import device as dv
    from tests.gpu_helpers import device_inputs, params_of
    q, k, v = device_inputs(prob)
    p = params_of(prob, cp, 1)
    plans, base = [], 0
    for r in rank_order:
        slabs, npairs = rlk.rlk_attn_plan_states(p, prob.cu_q, prob.cu_k, r, base)
        plans.append((r, slabs, base))
        base += npairs
    so = torch.empty((base, 128), dtype=torch.float32, device="cuda")
    sl = torch.empty((base,), dtype=torch.float32, device="cuda")
    for r, slabs, b0 in plans:
        rlk.rlk_attn_prefill_states(p, q, k, v, prob.cu_q, prob.cu_k, r, b0, so, sl)
    slabs = np.concatenate([s for _, s, _ in plans])
    slabs = slabs[np.random.default_rng(shuffle_seed).permutation(len(slabs))]
    return p, dv.slabs_to_device(slabs), len(slabs), so, sl, q.shape[0]


def test_noalloc_merge_matches_workspace_merge_twice():
    from tests.gpu_helpers import TOL_LSE, TOL_OUT, empty_outputs, lib, to_np, torch_cuda
    torch = torch_cuda()
    rlk = lib()
    for prob, cp, order, seed in [
        (synth.prefill_problem(lens=[300, 129, 1000, 17], hq=32, hkv=8, block=128, seed=41), 4, [2, 0, 3, 1], 1),
        (synth.prefill_problem(lens=[256], hq=32, hkv=8, block=64, seed=42), 2, [1, 0], 2),
    ]:
        p, dslabs, n, so, sl, rows = _tables(prob, cp, order, seed)
        ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, prob.cu_q, prob.cu_k), dtype=torch.uint8,
                         device="cuda")
        ref = empty_outputs(torch, rows, prob.hq)
        rlk.rlk_attn_merge_states(p, prob.cu_q, prob.cu_k, dslabs, n, so, sl, *ref, ws)
        ref = to_np(*ref)
        for _ in range(2):
            got = empty_outputs(torch, rows, prob.hq)
            rlk.rlk_attn_merge_states_noalloc(p, prob.cu_q, prob.cu_k, dslabs, n, so, sl, *got)
            rlk.rlk_attn_check_device_error()
            got = to_np(*got)
            assert np.abs(got[0] - ref[0]).max() <= TOL_OUT
            assert np.abs(got[2] - ref[2]).max() <= TOL_LSE
            assert np.array_equal(got[0].view(np.uint32), ref[0].view(np.uint32))
            assert np.array_equal(got[1].view(np.uint32), ref[1].view(np.uint32))
            assert np.array_equal(got[2].view(np.uint32), ref[2].view(np.uint32))


def test_noalloc_merge_at_the_scratch_limit():
    # num_seqs * max blocks == the 65,536-entry scratch exactly: 16 one-token
    # queries over 262,144 keys each, KV block 64 (4,096 blocks per
    # sequence), Hq = Hkv = 1.  The states are filled on the host (the merge
    # only reads the table), the slabs arrive permuted, and the no-alloc
    # merge must give the workspace merge's bits on two calls in a row.
    from tests.gpu_helpers import empty_outputs, lib, to_np, torch_cuda
    import deterministic_context_attention_gb300 as rlk_mod
    from deterministic_context_attention_gb300 import device as dv
    torch = torch_cuda()
    rlk = lib()
    n_seq, kv_len, block = 16, 262144, 64
    nb = kv_len // block
    assert n_seq * nb == 65536
    cu_q = np.arange(n_seq + 1, dtype=np.int32)
    cu_k = (np.arange(n_seq + 1, dtype=np.int64) * kv_len).astype(np.int32)
    p = rlk.make_params(n_seq, 1, 1, block)
    n_pairs = n_seq * nb
    rng = np.random.default_rng(61)
    so = torch.from_numpy(rng.standard_normal((n_pairs, 128), dtype=np.float32)).cuda()
    sl = torch.from_numpy((3.0 * rng.standard_normal(n_pairs)).astype(np.float32)).cuda()
    slabs = np.zeros(n_pairs, dtype=rlk_mod.SLAB_DTYPE)
    slabs["seq"] = np.repeat(np.arange(n_seq), nb)
    slabs["block"] = np.tile(np.arange(nb), n_seq)
    slabs["row_begin"] = 0
    slabs["row_count"] = 1
    slabs["offset"] = np.arange(n_pairs)
    slabs = slabs[rng.permutation(n_pairs)]
    dslabs = dv.slabs_to_device(slabs)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, cu_q, cu_k), dtype=torch.uint8, device="cuda")
    ref = empty_outputs(torch, n_seq, 1)
    rlk.rlk_attn_merge_states(p, cu_q, cu_k, dslabs, n_pairs, so, sl, *ref, ws)
    rlk.rlk_attn_check_device_error()
    ref = to_np(*ref)
    assert np.isfinite(ref[0]).all() and np.isfinite(ref[2]).all()
    for _ in range(2):
        got = empty_outputs(torch, n_seq, 1)
        rlk.rlk_attn_merge_states_noalloc(p, cu_q, cu_k, dslabs, n_pairs, so, sl, *got)
        rlk.rlk_attn_check_device_error()
        got = to_np(*got)
        for a, b in zip(got, ref):
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
