"""Host-side checks of the C ABI (no GPU): the library loads and exports every
entry point include/rlk_attn.h declares, argument validation fails closed
before any launch, and the block plan / CP partition / manifest hash behave
as the pages fix them."""
import ctypes
import os
import re

import math

import numpy as np
import pytest

import deterministic_context_attention_gb300 as rlk
from deterministic_context_attention_gb300 import build as rbuild
from deterministic_context_attention_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "rlk_attn.h")


@pytest.fixture(scope="module")
def lib():
    rbuild.build()
    return rlk.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"\b(rlk_attn_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_symbols()
    assert len(names) >= 11
    for n in names:
        assert hasattr(lib, n), n
    assert "global_block_index" in rlk.rlk_attn_core_id()


def test_slab_struct_layout_matches_header():
    assert rlk.SLAB_DTYPE.itemsize == 32
    assert ctypes.sizeof(rlk.rlk_attn_params) == 36


@pytest.mark.parametrize("layout", [rlk.CONTIGUOUS, rlk.ZIGZAG])
@pytest.mark.parametrize("cp", [1, 2, 4, 8])
def test_plan_covers_every_block_once(lib, cp, layout):
    lens = [4096, 3000, 1024, 777]
    cu = synth.cu_seqlens(lens)
    p = rlk.make_params(4, cp_size=cp, cp_layout=layout)
    all_slabs, all_pairs = rlk.rlk_attn_plan_states(p, cu, cu, -1, 0)
    assert len(all_slabs) == 32 + 24 + 8 + 7
    seen = {}
    base = 0
    for r in range(cp):
        slabs, npairs = rlk.rlk_attn_plan_states(p, cu, cu, r, base)
        for s in slabs:
            key = (int(s["seq"]), int(s["block"]))
            assert key not in seen
            seen[key] = r
            assert s["producer"] == r
        if len(slabs):
            assert slabs["offset"][0] == base
        base += npairs
    assert base == all_pairs
    assert sorted(seen) == sorted((int(s["seq"]), int(s["block"])) for s in all_slabs)
    # rows of each slab: those whose causal window reaches the block
    for s in all_slabs:
        assert s["row_begin"] == s["block"] * 128
        assert s["row_count"] == lens[s["seq"]] - s["row_begin"]
    # (row, block) pairs of the 4-sequence workload, times 32 heads
    pairs = sum(sum(L - b * 128 for b in range((L + 127) // 128)) for L in lens)
    assert all_pairs == pairs * 32


def test_plan_chunked_rows_are_bottom_right(lib):
    # 100 new queries over a cache of 1000 keys: every query sees blocks 0..7
    cu_q = np.array([0, 100], np.int32)
    cu_k = np.array([0, 1000], np.int32)
    p = rlk.make_params(1, num_q_heads=16, num_kv_heads=4)
    slabs, npairs = rlk.rlk_attn_plan_states(p, cu_q, cu_k)
    assert len(slabs) == 8
    # block 7 holds keys 896..999; query row i sits at 900 + i
    assert slabs[-1]["row_begin"] == 0 and slabs[-1]["row_count"] == 100
    assert npairs == 8 * 100 * 16


def test_manifest_hash_depends_on_blocks_and_producers(lib):
    cu = synth.cu_seqlens([4096, 3000, 1024, 777])
    h1 = rlk.rlk_attn_block_manifest_hash(rlk.make_params(4, cp_size=2), cu, cu)
    assert h1 == rlk.rlk_attn_block_manifest_hash(rlk.make_params(4, cp_size=2), cu, cu)
    assert h1 != rlk.rlk_attn_block_manifest_hash(rlk.make_params(4, cp_size=4), cu, cu)
    assert h1 != rlk.rlk_attn_block_manifest_hash(rlk.make_params(4, cp_size=2, kv_block_size=64), cu, cu)


@pytest.mark.parametrize("field,value,status", [
    ("head_dim", 64, 2), ("causal", 0, 2), ("kv_block_size", 32, 2), ("cp_size", 9, 1),
    ("num_kv_heads", 3, 1), ("num_seqs", 0, 2), ("softmax_scale", float("nan"), 1),
])
def test_bad_params_fail_closed(lib, field, value, status):
    cu = synth.cu_seqlens([16])
    p = rlk.make_params(1)
    setattr(p, field, value)
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_prefill(p, 16, 16, 16, cu, cu, -1, 16, None, 16, stream=0)
    assert e.value.status == status
    assert rlk.rlk_attn_last_error()


def test_bad_lengths_and_pointers_fail_closed(lib):
    p = rlk.make_params(1)
    with pytest.raises(rlk.RlkError) as e:  # q_len > kv_len
        rlk.rlk_attn_prefill(p, 16, 16, 16, [0, 20], [0, 10], -1, 16, None, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(rlk.RlkError) as e:  # misaligned q
        rlk.rlk_attn_prefill(p, 18, 16, 16, [0, 10], [0, 10], -1, 16, None, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(rlk.RlkError) as e:  # no output
        rlk.rlk_attn_prefill(p, 16, 16, 16, [0, 10], [0, 10], -1, None, None, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(rlk.RlkError) as e:  # cp_rank out of range
        rlk.rlk_attn_prefill(p, 16, 16, 16, [0, 10], [0, 10], 1, 16, None, 16, stream=0)
    assert e.value.status == 1
    with pytest.raises(rlk.RlkError) as e:  # page size that does not divide the block
        rlk.rlk_attn_decode_paged(p, 16, 16, 16, 4, 12, 16, 4, [10], 16, None, 16, stream=0)
    assert e.value.status == 2
    with pytest.raises(rlk.RlkError) as e:  # context longer than its page table row
        rlk.rlk_attn_decode_paged(p, 16, 16, 16, 4, 16, 16, 4, [65], 16, None, 16, stream=0)
    assert e.value.status == 1


def test_workspace_sizes(lib):
    cu = synth.cu_seqlens([4096, 3000, 1024, 777])
    p = rlk.make_params(4)
    assert rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, cu, cu) >= 4 * 32 * 4
    assert rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_BACKWARD, cu) >= int(cu[-1]) * 32 * 4
    assert rlk.rlk_attn_workspace_size(p, 99, cu, cu) == 0
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_merge_states(p, cu, cu, 16, 1, 16, 16, 16, None, 16, 16, 8, stream=0, n_state_pairs=1)
    assert e.value.status == 3


def test_noalloc_merge_rejects_oversized_problem_before_any_device_work(lib):
    # 128 sequences of 262,144 keys: 128 * 2048 blocks is 4x the 65,536-entry
    # scratch; the entry point must refuse before it touches the device (the
    # pointers below are placeholders that are never dereferenced)
    cu = synth.cu_seqlens([262144] * 128)
    p = rlk.make_params(128)
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_merge_states_noalloc(p, cu, cu, 16, 1, 16, 16, 16, None, 16, stream=0, n_state_pairs=1)
    assert e.value.status == 2
    assert "scratch" in rlk.rlk_attn_last_error()


def test_split_decode_rejects_before_any_launch(lib):
    # every case below fails validation on the host, before the library
    # touches the device, so placeholder pointers never reach a kernel
    p = rlk.make_params(1)
    for k in (-1, 65):  # split_k outside 0..64
        with pytest.raises(rlk.RlkError) as e:
            rlk.rlk_attn_decode_paged_splitk(p, 16, 16, 16, 4, 16, 16, 4, [10], k, 16, None, 16, 16, 1 << 20,
                                             stream=0)
        assert e.value.status == 1
    with pytest.raises(rlk.RlkError) as e:  # workspace smaller than the state table
        rlk.rlk_attn_decode_paged_splitk(p, 16, 16, 16, 4, 16, 16, 4, [10], 2, 16, None, 16, 16, 64, stream=0)
    assert e.value.status == 3
    p64 = rlk.make_params(1, kv_block_size=64)
    with pytest.raises(rlk.RlkError) as e:  # 64-key blocks: the transposed kernel takes 128
        rlk.rlk_attn_decode_paged_splitk(p64, 16, 16, 16, 4, 16, 16, 4, [10], 2, 16, None, 16, 16, 1 << 20,
                                         stream=0)
    assert e.value.status == 2
    pg = rlk.make_params(1, num_q_heads=32, num_kv_heads=2)
    with pytest.raises(rlk.RlkError) as e:  # 16 query heads per KV head
        rlk.rlk_attn_decode_paged_splitk(pg, 16, 16, 16, 4, 16, 16, 4, [10], 2, 16, None, 16, 16, 1 << 20,
                                         stream=0)
    assert e.value.status == 2


def test_split_decode_workspace_size(lib):
    p = rlk.make_params(2)  # Hq 32
    # 300 and 129 tokens: 3 + 2 blocks of 128; 516 bytes per (block, query
    # head), rounded up to 256, then 64 8-byte fill flags per (sequence, KV head)
    got = rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, [300, 129])
    assert got == (5 * 32 * 129 * 4 + 255) // 256 * 256 + 2 * 8 * 64 * 8
    assert rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_DECODE_SPLIT, None, [300, 0]) == 0


def test_decode_auto_split_choice(lib):
    # host-only policy query: few long sequences spread over the SMs, a batch
    # that already fills them stays single-pass
    p4 = rlk.make_params(4)  # Hq 32 / Hkv 8: 32 (sequence, KV head) pairs
    # few pairs: the largest k whose items and fold CTAs (one warp per
    # (sequence, query head), 15 a CTA) are resident at once, one per SM:
    # 32 pairs x 4 + ceil(128 / 15) = 137 <= 152, 32 x 5 + 9 > 152
    assert rlk.rlk_attn_decode_auto_split(p4, [32768] * 4, 152) == 4
    assert rlk.rlk_attn_decode_auto_split(p4, [128] * 4, 152) == 1  # one block each: nothing to split
    p64 = rlk.make_params(64)
    assert rlk.rlk_attn_decode_auto_split(p64, [32768] * 64, 152) == 1  # 512 pairs already cover 152 SMs
    p1 = rlk.make_params(1)
    assert rlk.rlk_attn_decode_auto_split(p1, [131072], 152) == 18  # 8 pairs x 18 + 3 fold CTAs = 147
    assert rlk.rlk_attn_decode_auto_split(p1, [131072], 1) == 1  # a single SM gains nothing from splitting
    assert rlk.rlk_attn_decode_auto_split(p4, [32768, 0, 5, 5], 152) == -1
    assert rlk.rlk_attn_decode_auto_split(p4, [32768] * 4, 0) == -1


def test_rope_table_values_and_validation(lib):
    t = rlk.rlk_attn_rope_table(1e6, 3)
    assert t.shape == (3, 128) and t.dtype == np.float32
    np.testing.assert_array_equal(t[0, :64], np.ones(64, np.float32))   # position 0: cos 0, sin 0
    np.testing.assert_array_equal(t[0, 64:], np.zeros(64, np.float32))
    assert t[1, 0] == np.float32(math.cos(1.0)) and t[1, 64] == np.float32(math.sin(1.0))
    f1 = 1e6 ** (-2.0 / 128)
    assert t[2, 1] == np.float32(math.cos(2 * f1)) and t[2, 65] == np.float32(math.sin(2 * f1))
    for theta, max_pos in ((1.0, 4), (float("inf"), 4), (1e6, 0)):
        with pytest.raises(rlk.RlkError) as e:
            rlk.rlk_attn_rope_table(theta, max_pos)
        assert e.value.status == 1


def test_rope_rejects_before_any_launch(lib):
    # every case fails host validation before the library touches the
    # device, so the placeholder pointers never reach a kernel
    p = rlk.make_params(2)
    cu = [0, 10, 20]
    bad = [
        dict(offs=[0, 95], max_pos=100),          # sequence 1 reaches position 104
        dict(offs=[-1, 0], max_pos=100),          # negative offset
        dict(x=17),                               # unaligned
        dict(heads=0),
        dict(cu=[1, 10, 20]),                     # does not start at 0
        dict(cu=[0, 10, 5]),                      # not monotone
        dict(table=None),
    ]
    for b in bad:
        with pytest.raises(rlk.RlkError) as e:
            rlk.rlk_attn_rope(p, b.get("x", 16), 16, b.get("heads", 8), b.get("cu", cu), b.get("offs", None),
                              b.get("table", 16), b.get("max_pos", 100), stream=0)
        assert e.value.status == 1, b


def test_decode_rope_rejects_before_any_launch(lib):
    def call(p, seqlens=(50,), table=16, max_pos=4096):
        rlk.rlk_attn_decode_paged_rope(p, 16, 16, 16, 4, 16, 16, 4, list(seqlens), table, max_pos, 16, None, 16,
                                       stream=0)
    p = rlk.make_params(1)
    for kw, status in ((dict(table=None), 1), (dict(max_pos=40), 1)):  # no table; position 49 past 40
        with pytest.raises(rlk.RlkError) as e:
            call(p, **kw)
        assert e.value.status == status
    for prm in (rlk.make_params(1, kv_block_size=64), rlk.make_params(1, num_q_heads=32, num_kv_heads=2)):
        with pytest.raises(rlk.RlkError) as e:  # the in-kernel RoPE lives in the transposed decode kernel only
            call(prm)
        assert e.value.status == 2


def test_split_decode_rope_rejects_before_any_launch(lib):
    p = rlk.make_params(1)

    def call(table=16, max_pos=4096, seqlens=(50,)):
        rlk.rlk_attn_decode_paged_splitk_rope(p, 16, 16, 16, 4, 16, 16, 4, list(seqlens), 2, table, max_pos, 16,
                                              None, 16, 16, 1 << 20, stream=0)
    for kw in (dict(table=None), dict(max_pos=40)):  # no table; position 49 past 40
        with pytest.raises(rlk.RlkError) as e:
            call(**kw)
        assert e.value.status == 1


def test_large_batch_validates_every_range_before_any_launch(lib):
    # 300 sequences run as ranges of 128; a context length of 0 in the third
    # range must fail the whole call in its host checks, before the library
    # touches the device (the tensor pointers are placeholders never read)
    p = rlk.make_params(300, 8, 2, 128)
    ctx = np.full(300, 64, np.int32)
    ctx[260] = 0
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_decode_paged(p, 16, 16, 16, 8, 16, 16, 4, ctx, 16, None, 16, stream=0)
    assert e.value.status == 1 and "sequence 4" in rlk.rlk_attn_last_error()  # index 260 is the 5th of range 2
    cu = synth.cu_seqlens([5] * 300)
    cuk = cu.copy()
    cuk[270:] += 3  # sequence 269 has a longer KV side: fine ...
    cq_bad = cu.copy()
    cq_bad[281:] += 10  # ... but sequence 280 has q_len 15 > kv_len 5
    with pytest.raises(rlk.RlkError) as e:
        rlk.rlk_attn_prefill(p, 16, 16, 16, cq_bad, cu, -1, 16, None, 16, stream=0)
    assert e.value.status == 1


def test_large_batch_plan_and_workspace(lib):
    # the host-side helpers take the whole batch: the plan's slabs keep the
    # batch's sequence ids and consecutive pair offsets
    lens = [3] * 200
    cu = synth.cu_seqlens(lens)
    p = rlk.make_params(200, 8, 2, 64)
    slabs, npairs = rlk.rlk_attn_plan_states(p, cu, cu, -1, 0)
    assert len(slabs) == 200 and npairs == 200 * 3 * 8
    assert list(slabs["seq"]) == list(range(200))
    assert np.all(np.diff(slabs["offset"]) == 24)
    assert rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, cu, cu) >= 200 * 4
