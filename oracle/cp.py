"""The oracle's own logical context-parallel (CP) bookkeeping -- TEST
INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Emulated CP follows "WS2 Attention PR5 Drift Benchmark" (Transformer Engine
Reuse: every rank builds partial states (out_i, lse_i, global_block_index_i);
the merge sorts them by global_block_index, whatever rank or arrival order
produced them) and "[WS2][Attention] H100 validation and reproduction guide"
(Status / Acceptance: full-KV arithmetic retained, so a state always covers a
whole global block; out/LSE bitwise equal across 2/4/8 ranks).

Partition of a sequence of n tokens over cp logical ranks (the pages name the
CP sizes but not the partition; the configs ask for contiguous halves and a
zigzag load-balanced split):
  * contiguous: cp chunks with bounds floor(c * n / cp); rank r owns chunk r.
  * zigzag: 2*cp chunks with bounds floor(c * n / (2 cp)); rank r owns chunks
    r and 2*cp - 1 - r.
The producer of global block b is the rank that owns its first key b*block.
"""
from __future__ import annotations

import numpy as np

from . import fold_f32, row_block_states_f64

CONTIGUOUS, ZIGZAG = 0, 1


def chunks(n: int, cp: int, layout: int):
    """List of (rank, begin, end) token chunks of one sequence."""
    if layout == CONTIGUOUS:
        bounds = [(c * n) // cp for c in range(cp + 1)]
        return [(c, bounds[c], bounds[c + 1]) for c in range(cp)]
    bounds = [(c * n) // (2 * cp) for c in range(2 * cp + 1)]
    out = []
    for c in range(2 * cp):
        rank = c if c < cp else 2 * cp - 1 - c
        out.append((rank, bounds[c], bounds[c + 1]))
    return out


def owner(pos: int, n: int, cp: int, layout: int) -> int:
    """Logical rank that owns token ``pos`` of a sequence of ``n`` tokens."""
    for rank, b, e in chunks(n, cp, layout):
        if b <= pos < e:
            return rank
    raise ValueError("position outside the sequence")


def block_producer(b: int, block: int, kv_len: int, cp: int, layout: int) -> int:
    return owner(b * block, kv_len, cp, layout)


def emulated_cp_fold(q, k, v, cu_q, cu_k, scale, block, cp, layout, token, head,
                     rank_order=None, reverse_within_rank=False):
    """Emulated CP merge of one (token, head).

    Each logical rank contributes the FP32 states of the global blocks it
    produces; states arrive rank by rank in ``rank_order`` (default 0..cp-1),
    each rank's states in ascending or reversed block order.  The canonical
    fold then sorts by global_block_index.  Returns (out [D] f32, lse f32,
    arrival gbi list).
    """
    o64, l64 = row_block_states_f64(q, k, v, cu_q, cu_k, scale, block, token, head)
    s = int(np.searchsorted(np.asarray(cu_q), token, side="right") - 1)
    kv_len = int(cu_k[s + 1] - cu_k[s])
    nb = o64.shape[0]
    per_rank = {r: [] for r in range(cp)}
    for b in range(nb):
        per_rank[block_producer(b, block, kv_len, cp, layout)].append(b)
    order = list(range(cp)) if rank_order is None else list(rank_order)
    arrival = []
    for r in order:
        bl = per_rank[r][::-1] if reverse_within_rank else per_rank[r]
        arrival.extend(bl)
    o32 = o64.astype(np.float32)[arrival]
    l32 = l64.astype(np.float32)[arrival]
    out, lse = fold_f32(np.array(arrival, np.int32), o32, l32)
    return out, lse, arrival
