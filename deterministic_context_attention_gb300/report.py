"""Machine-readable drift report of the deterministic attention path.

Runs the library's entry points on a synthetic workload and records, per
case, the drift classes of "WS2 Attention PR5 Drift Benchmark" (drift-class
table) in this library's own schema ``rlk_attn_cp_drift/v1``:

* ``drift.cp_merge_fp32`` -- max |out_f32(candidate) - out_f32(CP=1 fused)|
  for logical CP sizes (fused row ownership and states + merge in permuted
  arrival) and chunked replay; the strict claim is 0.0;
* ``drift.dtype_path_vs_fp32`` -- max |out_bf16 - out_f32| (the final-write
  rounding; nonzero by construction);
* ``merge_order_probe`` -- max |merge(reversed arrival) - merge(sorted)|;
  strict 0.0;
* ``backward`` -- max |dQ/dK/dV(CP=r) - dQ/dK/dV(CP=1)|; strict 0.0;
* ``drift.dlogp`` -- the active-token log-probability drift: each output row
  (all heads, FP32) is projected through a seeded synthetic FP32 lm_head
  (the pages' dlogp check, "[WS2][Attention] H100 validation and
  reproduction guide", Status: Out/LSE/dlogp max abs 0.0) and the
  log-probability of a seeded token per row is compared with the CP=1
  fused path's; strict 0.0.

Each case records its topology, the block size, the block manifest hash and
per-logical-rank counts; the root records ``merge_order`` =
global_block_index and ``downcast_at`` = final_write (Report Contract).

    python -m deterministic_context_attention_gb300.report [--output PATH] [--small]
"""
from __future__ import annotations

import argparse
import json
import sys

import numpy as np

from . import synth

SCHEMA = "rlk_attn_cp_drift/v1"


def _dlogp(out, vocab=512, seed=7):
    """Log-probability of a seeded token per row after a seeded FP32 lm_head
    (N(0, 1/width)) over the row's outputs of all heads; FP32 throughout,
    the same numpy arithmetic for every path compared."""
    rows = out.shape[0]
    x = np.ascontiguousarray(out.reshape(rows, -1), dtype=np.float32)
    w, tok = synth.lm_head(x.shape[1], rows, vocab, seed)
    logits = x @ w
    m = logits.max(axis=1, keepdims=True)
    lse = m[:, 0] + np.log(np.exp(logits - m).sum(axis=1, dtype=np.float32), dtype=np.float32)
    return logits[np.arange(rows), tok] - lse


def _maxabs(a, b):
    return float(np.max(np.abs(np.asarray(a, np.float64) - np.asarray(b, np.float64)))) if np.size(a) else 0.0


def drift_report(lens=(4096, 3000, 1024, 777), hq=32, hkv=8, block=128, seed=1, rope=True,
                 cp_sizes=(2, 4, 8), chunk_sizes=(512, 2048), backward_lens=(1024, 512),
                 backward_cp=(2, 4)):
    import torch

    import deterministic_context_attention_gb300 as rlk
    from .build import build
    from . import device as dv

    build()
    rlk.load()
    prob = synth.prefill_problem(list(lens), hq=hq, hkv=hkv, block=block, seed=seed, rope=rope)
    q, k, v = dv.bf16_to_device(prob.q), dv.bf16_to_device(prob.k), dv.bf16_to_device(prob.v)
    rows = q.shape[0]

    def outputs():
        return (torch.empty((rows, hq, 128), dtype=torch.float32, device="cuda"),
                torch.empty((rows, hq, 128), dtype=torch.bfloat16, device="cuda"),
                torch.empty((rows, hq), dtype=torch.float32, device="cuda"))

    def fused(cp, layout, ranks):
        o, ob, l = outputs()
        p = rlk.make_params(len(lens), hq, hkv, block, cp, layout, prob.scale)
        for r in ranks:
            rlk.rlk_attn_prefill(p, q, k, v, prob.cu_q, prob.cu_k, r, o, ob, l)
        rlk.rlk_attn_check_device_error()
        return o.cpu().numpy(), ob.float().cpu().numpy(), l.cpu().numpy()

    def states_merge(cp, layout, order, reverse):
        p = rlk.make_params(len(lens), hq, hkv, block, cp, layout, prob.scale)
        plans, base = [], 0
        for r in order:
            slabs, n = rlk.rlk_attn_plan_states(p, prob.cu_q, prob.cu_k, r, base)
            plans.append((r, slabs, base))
            base += n
        so = torch.empty((base, 128), dtype=torch.float32, device="cuda")
        sl = torch.empty((base,), dtype=torch.float32, device="cuda")
        for r, slabs, b0 in plans:
            rlk.rlk_attn_prefill_states(p, q, k, v, prob.cu_q, prob.cu_k, r, b0, so, sl)
        slabs = np.concatenate([s for _, s, _ in plans])
        if reverse:
            slabs = slabs[::-1].copy()
        ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, prob.cu_q, prob.cu_k),
                         dtype=torch.uint8, device="cuda")
        o, ob, l = outputs()
        rlk.rlk_attn_merge_states(p, prob.cu_q, prob.cu_k, dv.slabs_to_device(slabs), len(slabs), so, sl, o, ob,
                                  l, ws)
        rlk.rlk_attn_check_device_error()
        per_rank = [{"rank": int(r), "states_slabs": int(len(s)),
                     "state_pairs": int(sum(int(x["row_count"]) for x in s) * hq)} for r, s, _ in plans]
        return (o.cpu().numpy(), ob.float().cpu().numpy(), l.cpu().numpy()), per_rank

    base = fused(1, rlk.ZIGZAG, [-1])
    base_dlogp = _dlogp(base[0])
    root = {"schema_version": SCHEMA, "core_id": rlk.rlk_attn_core_id(),
            "merge_order": "global_block_index", "downcast_at": "final_write",
            "target": {"heads_q": hq, "heads_kv": hkv, "head_dim": 128, "kv_block": block,
                       "lens": list(lens), "rope": {"theta": 1.0e6, "style": "rotate_half"} if rope else None,
                       "seed": seed},
            "cases": []}
    sorted_merge, _ = states_merge(1, rlk.ZIGZAG, [0], False)
    reversed_merge, _ = states_merge(1, rlk.ZIGZAG, [0], True)
    root["merge_order_probe"] = {"max_abs_out": _maxabs(reversed_merge[0], sorted_merge[0]),
                                 "max_abs_lse": _maxabs(reversed_merge[2], sorted_merge[2])}
    for cp in cp_sizes:
        for layout, lname in ((rlk.ZIGZAG, "zigzag"), (rlk.CONTIGUOUS, "contiguous")):
            order = list(np.random.default_rng(cp).permutation(cp))
            f = fused(cp, layout, order)
            sm, per_rank = states_merge(cp, layout, order[::-1], True)
            p = rlk.make_params(len(lens), hq, hkv, block, cp, layout, prob.scale)
            root["cases"].append({
                "mode": "full_prefill", "topology": {"tp": 1, "cp": cp, "layout": lname},
                "split_kv_policy": f"fixed global blocks of {block} keys",
                "block_manifest_hash": f"{rlk.rlk_attn_block_manifest_hash(p, prob.cu_q, prob.cu_k):016x}",
                "drift": {"cp_merge_fp32": max(_maxabs(f[0], base[0]), _maxabs(sm[0], base[0])),
                          "lse": max(_maxabs(f[2], base[2]), _maxabs(sm[2], base[2])),
                          "dlogp": max(_maxabs(_dlogp(f[0]), base_dlogp), _maxabs(_dlogp(sm[0]), base_dlogp)),
                          "dtype_path_vs_fp32": _maxabs(f[1], f[0])},
                "per_logical_cp_rank": per_rank})
    # chunked replay: each sequence's queries in chunks against the growing cache
    for chunk in chunk_sizes:
        o, ob, l = outputs()
        p = rlk.make_params(1, hq, hkv, block, 1, rlk.ZIGZAG, prob.scale)
        for s in range(len(lens)):
            q0, q1, k0 = int(prob.cu_q[s]), int(prob.cu_q[s + 1]), int(prob.cu_k[s])
            for c0 in range(0, q1 - q0, chunk):
                c1 = min(c0 + chunk, q1 - q0)
                rlk.rlk_attn_prefill(p, q[q0 + c0:q0 + c1], k[k0:k0 + c1], v[k0:k0 + c1], [0, c1 - c0], [0, c1], -1,
                                     o[q0 + c0:q0 + c1], ob[q0 + c0:q0 + c1], l[q0 + c0:q0 + c1])
        rlk.rlk_attn_check_device_error()
        on = o.cpu().numpy()
        root["cases"].append({"mode": "chunked_prefill", "chunk": chunk, "topology": {"tp": 1, "cp": 1},
                              "drift": {"cp_merge_fp32": _maxabs(on, base[0]),
                                        "lse": _maxabs(l.cpu().numpy(), base[2]),
                                        "dlogp": _maxabs(_dlogp(on), base_dlogp)}})
    # backward drift across logical CP sizes
    bprob = synth.prefill_problem(list(backward_lens), hq=hq, hkv=hkv, block=128, seed=seed + 3)
    bq, bk, bv = dv.bf16_to_device(bprob.q), dv.bf16_to_device(bprob.k), dv.bf16_to_device(bprob.v)
    T = bq.shape[0]
    pb = rlk.make_params(len(backward_lens), hq, hkv, 128, 1, rlk.ZIGZAG, bprob.scale)
    bo = torch.empty((T, hq, 128), dtype=torch.float32, device="cuda")
    bl = torch.empty((T, hq), dtype=torch.float32, device="cuda")
    rlk.rlk_attn_prefill(pb, bq, bk, bv, bprob.cu_q, bprob.cu_k, -1, bo, None, bl)
    do = dv.bf16_to_device(synth.normal_bf16(seed + 3, synth.T_DOUT, bprob.q.shape))

    def grads(cp, ranks):
        p = rlk.make_params(len(backward_lens), hq, hkv, 128, cp, rlk.ZIGZAG, bprob.scale)
        g = [torch.empty((T, h, 128), dtype=torch.float32, device="cuda") for h in (hq, hkv, hkv)]
        ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_BACKWARD, bprob.cu_q), dtype=torch.uint8,
                         device="cuda")
        for r in ranks:
            rlk.rlk_attn_backward(p, bq, bk, bv, bo, do, bl, bprob.cu_q, r, g[0], g[1], g[2], ws)
        rlk.rlk_attn_check_device_error()
        return [x.cpu().numpy() for x in g]

    g1 = grads(1, [-1])
    for cp in backward_cp:
        gc = grads(cp, list(range(cp))[::-1])
        root["cases"].append({"mode": "backward", "topology": {"tp": 1, "cp": cp, "layout": "zigzag"},
                              "lens": list(backward_lens),
                              "backward": {n: _maxabs(a, b) for n, a, b in zip(("dq", "dk", "dv"), gc, g1)}})
    strict = [c["drift"]["cp_merge_fp32"] for c in root["cases"] if "drift" in c]
    strict += [c["drift"]["lse"] for c in root["cases"] if "drift" in c]
    strict += [c["drift"]["dlogp"] for c in root["cases"] if "drift" in c]
    strict += [x for c in root["cases"] if "backward" in c for x in c["backward"].values()]
    strict += list(root["merge_order_probe"].values())
    root["strict_max_abs"] = max(strict) if strict else 0.0
    root["passed"] = root["strict_max_abs"] == 0.0
    return root


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--output", default=None)
    ap.add_argument("--small", action="store_true", help="a small workload (seconds)")
    a = ap.parse_args(argv)
    if a.small:
        rep = drift_report(lens=(300, 129, 1000, 17), cp_sizes=(2, 4), chunk_sizes=(7, 200),
                           backward_lens=(300, 129))
    else:
        rep = drift_report()
    text = json.dumps(rep, indent=1)
    if a.output:
        with open(a.output, "w") as f:
            f.write(text)
    print(json.dumps({"schema_version": rep["schema_version"], "passed": rep["passed"],
                      "strict_max_abs": rep["strict_max_abs"], "cases": len(rep["cases"])}))
    return 0 if rep["passed"] else 1


if __name__ == "__main__":
    sys.exit(main())
