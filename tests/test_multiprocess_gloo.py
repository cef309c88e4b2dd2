"""World-size-2 process-group checks on CPU (gloo): the host-side logic the
multi-rank paths use.

* Each process plans the partial states of its own logical CP rank with the
  library's host planner, storage bases from an exclusive scan of the ranks'
  pair counts; the gathered plans must cover every global block exactly once
  with disjoint, contiguous storage, and every rank must agree on the block
  manifest hash ("WS2 Attention PR5 Drift Benchmark", Report Contract: block
  metadata hash; Transformer Engine Reuse: states from every rank, merged by
  global_block_index).
* bench.py's max-over-ranks timing reduction returns the slowest rank's time
  on every rank.
"""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

LENS = [4096, 3000, 1024, 777]


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import deterministic_context_attention_gb300 as rlk
        from deterministic_context_attention_gb300 import synth
        import bench
        cu = synth.cu_seqlens(LENS)
        p = rlk.make_params(4, cp_size=world, cp_layout=rlk.ZIGZAG)
        _, my_pairs = rlk.rlk_attn_plan_states(p, cu, cu, rank, 0)
        counts = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(counts, torch.tensor([my_pairs], dtype=torch.int64))
        base = int(sum(int(c.item()) for c in counts[:rank]))
        slabs, _ = rlk.rlk_attn_plan_states(p, cu, cu, rank, base)
        raw = torch.from_numpy(slabs.view(np.uint8).copy())
        sizes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(sizes, torch.tensor([raw.numel()], dtype=torch.int64))
        mx = int(max(int(s.item()) for s in sizes))
        buf = torch.zeros(mx, dtype=torch.uint8)
        buf[:raw.numel()] = raw
        gathered = [torch.zeros(mx, dtype=torch.uint8) for _ in range(world)]
        dist.all_gather(gathered, buf)
        h = rlk.rlk_attn_block_manifest_hash(p, cu, cu)
        hashes = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(hashes, torch.tensor([h & 0x7FFFFFFFFFFFFFFF], dtype=torch.int64))
        slow = bench.max_over_ranks(10.0 + rank, dist)
        if rank == 0:
            allslabs = np.concatenate([g[:int(s.item())].numpy().view(rlk.SLAB_DTYPE)
                                       for g, s in zip(gathered, sizes)])
            np.save(os.path.join(out_dir, "slabs.npy"), allslabs)
            np.save(os.path.join(out_dir, "meta.npy"),
                    np.array([len(set(int(x.item()) for x in hashes)), slow, sum(int(c.item()) for c in counts)]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_two_rank_cp_plan_covers_blocks_once(tmp_path, world):
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn")
    import deterministic_context_attention_gb300 as rlk
    from deterministic_context_attention_gb300 import synth
    slabs = np.load(tmp_path / "slabs.npy")
    n_hash_values, slow, total_pairs = np.load(tmp_path / "meta.npy")
    assert n_hash_values == 1          # every rank computed the same manifest hash
    assert slow == 10.0 + world - 1    # the slowest rank's time reached every rank
    keys = sorted((int(s["seq"]), int(s["block"])) for s in slabs)
    assert keys == sorted(set(keys))
    assert len(keys) == sum((L + 127) // 128 for L in LENS)
    # storage: disjoint and contiguous over all ranks
    spans = sorted((int(s["offset"]), int(s["offset"]) + int(s["row_count"]) * 32) for s in slabs)
    assert spans[0][0] == 0 and spans[-1][1] == total_pairs
    for (a0, a1), (b0, b1) in zip(spans, spans[1:]):
        assert a1 == b0
    # the single-process plan of all ranks lists the same (seq, block) set
    cu = synth.cu_seqlens(LENS)
    full, _ = rlk.rlk_attn_plan_states(rlk.make_params(4, cp_size=world), cu, cu, -1, 0)
    assert keys == sorted((int(s["seq"]), int(s["block"])) for s in full)
