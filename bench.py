"""Benchmark: causal GQA prefill TFLOP/s (headline) plus paged-decode and
merge GB/s, on the synthetic Qwen3-8B attention workloads, against the
measured GB300 rooflines.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

A step is one fused causal prefill (rlk_attn_prefill) over the varlen batch
{4096, 3000, 1024, 777} tokens, Hq=32, Hkv=8, D=128, KV block 128, with the
inputs resident in HBM; L2 is flushed (a 512 MB write) before every timed
step and each step is timed with CUDA events on the launch stream.  `value`
is algorithmic TFLOP/s = 4*D*Hq*sum(visible (row, key) pairs) / time.  `e2e`
is the same metric through the public API from pinned host buffers
(host->device copy of q/k/v, the prefill, device->host copy of the same
outputs as the headline -- out_f32, out_bf16 and lse -- every step) over K
pipelined steps: uploads, compute and downloads on
three streams with double-buffered device tensors, as a serving loop would
run them.  Under torchrun every rank runs the same batch
on its own GPU (weak scaling, no collective on the data path).

Rank 0 adds, outside the timed region of the headline, one object per other
path (each with its own CUDA-event timing and L2 flush): "merge" (the
canonical fold of the prefill's CP=1 state table), "states" (the state
producer), "decode" (64 sequences, contexts U[512, 32768], 16-token pages),
"decode_long" (4 x 32768 tokens: single pass against the split decode),
"rope" (the RoPE pass over the prefill's Q and K in one launch, also after a
flush that leaves L2 clean), "prefill_rope" (the headline prefill with the
queries' RoPE inside the kernel), "backward" (2 x 4096) and "chunked" (2 x 8192 in chunks of
2048); --no-extras skips them.  --profile NAME runs one path a few times,
untimed, for ncu.

--impl reference times the CPU oracle (FP64 definition) on the host cores on
a bounded sample of the same workload's rows, in the same metric.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from deterministic_context_attention_gb300 import synth  # noqa: E402

METRIC = "causal prefill TFLOP/s + paged decode GB/s (% GB300 roofline), bit-invariant"
WORKLOAD = ("qwen3-8b causal GQA prefill, varlen {4096,3000,1024,777} (8897 tokens), Hq=32 Hkv=8 D=128, "
            "bf16 q/k/v N(0,1) + RoPE theta=1e6, KV block 128, logical CP=1, out fp32+bf16 + lse")


def kernel_traffic(name):
    """DRAM bytes per launch of a kernel from the committed ncu summary
    (profiles/traffic.json), or None when the kernel sources changed since
    the counters were taken."""
    import hashlib
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    entry = json.load(open(path))["kernels"].get(name)
    if not entry:
        return None
    h = hashlib.sha256()
    for src in entry["sources"]:
        h.update(open(os.path.join(ROOT, src), "rb").read())
    return entry["traffic_bytes"] if h.hexdigest() == entry["sources_sha256"] else None


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        d = json.load(open(path))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


def prefill_workload():
    cfg = dict(synth.CFG_PREFILL)
    prob = synth.prefill_problem(**cfg)
    flops = synth.prefill_flops(prob.cu_q, prob.cu_k, prob.hq, prob.d)
    return prob, flops


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            # raw samples go to RLK_BENCH_CLOCKS_DIR (default: the temp directory);
            # the JSON line carries their summary
            d = os.environ.get("RLK_BENCH_CLOCKS_DIR") or tempfile.gettempdir()
            os.makedirs(d, exist_ok=True)
            self.path = os.path.join(d, f"clocks_bench_{os.getpid()}.csv")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step device time (ms) of fn() with an L2 flush before each step.
    A short device-side sleep after the flush keeps the stream busy while the
    host prepares the launch, so host-side launch cost stays outside the
    events."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    for i in range(steps):
        flush.zero_()
        torch.cuda._sleep(400000)
        starts[i].record(stream)
        fn()
        ends[i].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def max_over_ranks(value, dist):
    """Largest value over the ranks of the default process group (the value
    itself without one).  The tensor lives where the backend wants it."""
    if dist is None or not dist.is_initialized():
        return float(value)
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(value)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_gpu(args):
    import torch
    import deterministic_context_attention_gb300 as rlk
    from deterministic_context_attention_gb300 import build as rbuild
    from deterministic_context_attention_gb300 import device as dv

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    if rank == 0 or world == 1:
        rbuild.build()
    if dist is not None:
        dist.barrier()
    rlk.load()
    peaks = load_peaks()
    stream = torch.cuda.current_stream()

    prob, flops = prefill_workload()
    q, k, v = dv.bf16_to_device(prob.q), dv.bf16_to_device(prob.k), dv.bf16_to_device(prob.v)
    rows = q.shape[0]
    p = rlk.make_params(4, 32, 8, 128, 1, rlk.ZIGZAG, prob.scale)
    out = torch.empty((rows, 32, 128), dtype=torch.float32, device="cuda")
    outb = torch.empty((rows, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows, 32), dtype=torch.float32, device="cuda")
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")

    def step():
        rlk.rlk_attn_prefill(p, q, k, v, prob.cu_q, prob.cu_k, -1, out, outb, lse, stream=stream)

    clocks = Clocks(local)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    t_wall0 = time.perf_counter()
    times = time_steps(torch, step, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t_wall0
    clk = clocks.stop()
    rlk.rlk_attn_check_device_error(stream)
    ms = max_over_ranks(float(np.mean(times)), dist)
    value = world * flops / (ms * 1e-3) / 1e12
    achieved = flops / (ms * 1e-3) / 1e12
    peak = peaks["bf16_tflops"]

    # ---- end to end through the public API from pinned host buffers: every
    # step copies its inputs host -> device, runs the prefill and copies its
    # outputs (FP32 and BF16 out and lse, the headline's output set) device ->
    # host.  Steps are pipelined the way a
    # serving loop double-buffers them: step i+1's upload (one stream) and
    # step i-1's download (another) overlap step i's compute, ordered by
    # events; the timed region spans all K steps, copies included.
    qh = torch.from_numpy(synth.bf16_bits(prob.q).view(np.int16)).pin_memory()
    kh = torch.from_numpy(synth.bf16_bits(prob.k).view(np.int16)).pin_memory()
    vh = torch.from_numpy(synth.bf16_bits(prob.v).view(np.int16)).pin_memory()
    out_h = [torch.empty((rows, 32, 128), dtype=torch.float32).pin_memory() for _ in range(2)]
    outb_h = [torch.empty((rows, 32, 128), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    lse_h = [torch.empty((rows, 32), dtype=torch.float32).pin_memory() for _ in range(2)]
    qd = [torch.empty_like(qh, device="cuda") for _ in range(2)]
    kd = [torch.empty_like(kh, device="cuda") for _ in range(2)]
    vd = [torch.empty_like(vh, device="cuda") for _ in range(2)]
    out_d = [torch.empty((rows, 32, 128), dtype=torch.float32, device="cuda") for _ in range(2)]
    outb_d = [torch.empty((rows, 32, 128), dtype=torch.bfloat16, device="cuda") for _ in range(2)]
    lse_d = [torch.empty((rows, 32), dtype=torch.float32, device="cuda") for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()

    def e2e_run(n):
        ev_in, ev_comp, ev_out = [], [], []
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(s_in)
        for i in range(n):
            b = i % 2
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_comp[i - 2])  # buffer b is free once step i-2 computed
                qd[b].copy_(qh, non_blocking=True)
                kd[b].copy_(kh, non_blocking=True)
                vd[b].copy_(vh, non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_in)
                ev_in.append(e)
            stream.wait_event(ev_in[i])
            if i >= 2:
                stream.wait_event(ev_out[i - 2])  # outputs b were read back
            rlk.rlk_attn_prefill(p, qd[b].view(torch.bfloat16), kd[b].view(torch.bfloat16), vd[b].view(torch.bfloat16),
                                 prob.cu_q, prob.cu_k, -1, out_d[b], outb_d[b], lse_d[b], stream=stream)
            e = torch.cuda.Event()
            e.record(stream)
            ev_comp.append(e)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_comp[i])
                out_h[b].copy_(out_d[b], non_blocking=True)
                outb_h[b].copy_(outb_d[b], non_blocking=True)
                lse_h[b].copy_(lse_d[b], non_blocking=True)
                e = torch.cuda.Event()
                e.record(s_out)
                ev_out.append(e)
        s_in.wait_event(ev_out[-1])
        t1.record(s_in)
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / n

    e2e_run(max(args.warmup, 2))
    e2e_ms = e2e_run(args.steps)
    rlk.rlk_attn_check_device_error(stream)
    h2d = (qh.numel() + kh.numel() + vh.numel()) * 2
    d2h = out_h[0].numel() * 4 + outb_h[0].numel() * 2 + lse_h[0].numel() * 4

    extras = {}
    if not args.no_extras and rank == 0:
        extras = measure_extras(torch, rlk, dv, peaks, prob, q, k, v, flush, stream, args)
        extras["prefill_rope"] = measure_prefill_rope(torch, rlk, peaks, prob, q, k, v, flush, stream, args, ms)

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic",
            "config": {"workload": WORKLOAD, "global_batch": 4 * world, "seq_len": "varlen 4096/3000/1024/777",
                       "parallelism": f"replicas{world}" if world > 1 else "single",
                       "l2": "flushed (512 MB write) before every timed step", "flops_per_step": flops},
            "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 3), "unit": "TFLOP/s",
                    "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
                    "ms_per_step": round(e2e_ms, 5), "outputs": "out_f32 + out_bf16 + lse (the headline's set)",
                    "pipeline": "double-buffered: upload of step i+1 and download of step i-1 overlap step i"},
            "gpu_launches": args.steps,
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak, "unit": "TFLOP/s",
                         "frac": round(achieved / peak, 4),
                         "traffic": kernel_traffic("rlk_fwd_kernel<128, fused>"),
                         "traffic_unit": "bytes per launch (ncu dram read + write)",
                         "peak_source": f"{peaks['source']} bf16 dense burst",
                         "kernel": "rlk_fwd_kernel<128, fused>",
                         "physical_frac": round(1.5 * achieved / peak, 4)},
            "clocks": clk,
            "wall_s_timed_region": round(wall, 3),
        }
        line.update(extras)
        if not args.no_cpu_baseline and world == 1:
            line["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def measure_extras(torch, rlk, dv, peaks, prob, q, k, v, flush, stream, args):
    """Paged decode GB/s and merge GB/s (each against the measured HBM
    roofline), states-producer and chunked-replay rates."""
    res = {}
    # ---- states (CP=1 plan) + merge on the prefill workload
    p = rlk.make_params(4, 32, 8, 128, 1, rlk.ZIGZAG, prob.scale)
    slabs, npairs = rlk.rlk_attn_plan_states(p, prob.cu_q, prob.cu_k, -1, 0)
    so = torch.empty((npairs, 128), dtype=torch.float32, device="cuda")
    sl = torch.empty((npairs,), dtype=torch.float32, device="cuda")
    ds = dv.slabs_to_device(slabs)
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, prob.cu_q, prob.cu_k), dtype=torch.uint8,
                     device="cuda")
    rows = q.shape[0]
    out = torch.empty((rows, 32, 128), dtype=torch.float32, device="cuda")
    outb = torch.empty((rows, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows, 32), dtype=torch.float32, device="cuda")
    t_states = time_steps(torch, lambda: rlk.rlk_attn_prefill_states(p, q, k, v, prob.cu_q, prob.cu_k, -1, 0, so,
                                                                      sl, stream=stream),
                          args.steps, args.warmup, flush, stream)
    t_merge = time_steps(torch, lambda: rlk.rlk_attn_merge_states(p, prob.cu_q, prob.cu_k, ds, len(slabs), so, sl,
                                                                   out, outb, lse, ws, stream=stream),
                         args.steps, args.warmup, flush, stream)
    rlk.rlk_attn_check_device_error(stream)
    merge_bytes = npairs * (128 * 4 + 4) + rows * 32 * (128 * 4 + 128 * 2 + 4) + len(slabs) * 32
    ms_m = float(np.mean(t_merge))
    ms_s = float(np.mean(t_states))
    gbs = merge_bytes / (ms_m * 1e-3) / 1e9
    res["merge"] = {"value": round(gbs, 1), "unit": "GB/s", "ms": round(ms_m, 4), "bytes": int(merge_bytes),
                    "frac": round(gbs / peaks["hbm_gbs"], 4), "peak": peaks["hbm_gbs"],
                    "note": "canonical fold of the CP=1 state table of the prefill workload (index kernel + fold kernel)"}
    states_bytes = npairs * (128 * 4 + 4)
    flops = synth.prefill_flops(prob.cu_q, prob.cu_k, 32, 128)
    res["states"] = {"tflops": round(flops / (ms_s * 1e-3) / 1e12, 2), "ms": round(ms_s, 4),
                     "write_gbs": round(states_bytes / (ms_s * 1e-3) / 1e9, 1), "state_bytes": int(states_bytes)}
    del so, sl
    torch.cuda.empty_cache()

    # ---- paged decode: 64 sequences, ctx ~ U[512, 32768], 16-token pages in a permuted pool
    g = torch.Generator(device="cuda")
    g.manual_seed(3)
    ctx = synth.rng(3, synth.T_LENS).integers(512, 32769, size=64).astype(np.int32)
    pages_per = (ctx + 15) // 16
    n_pages = int(pages_per.sum())
    perm = synth.rng(3, synth.T_PAGES).permutation(n_pages).astype(np.int32)
    max_pages = int(pages_per.max())
    pt = np.full((64, max_pages), -1, np.int32)
    off = 0
    for s in range(64):
        pt[s, :pages_per[s]] = perm[off:off + pages_per[s]]
        off += pages_per[s]
    kp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    vp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    qd = torch.randn((64, 32, 128), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    ptd = dv.i32_to_device(pt)
    pd = rlk.make_params(64, 32, 8, 128)
    dout = torch.empty((64, 32, 128), dtype=torch.float32, device="cuda")
    doutb = torch.empty((64, 32, 128), dtype=torch.bfloat16, device="cuda")
    dlse = torch.empty((64, 32), dtype=torch.float32, device="cuda")
    t_dec = time_steps(torch, lambda: rlk.rlk_attn_decode_paged(pd, qd, kp, vp, n_pages, 16, ptd, max_pages, ctx, dout,
                                                                 doutb, dlse, stream=stream),
                       args.steps, args.warmup, flush, stream)
    rlk.rlk_attn_check_device_error(stream)
    dec_bytes = int(ctx.astype(np.int64).sum()) * 8 * 128 * 2 * 2 + 64 * 32 * 128 * (2 + 4 + 2) + 64 * 32 * 4 \
        + int(pages_per.sum()) * 4
    ms_d = float(np.mean(t_dec))
    gbs = dec_bytes / (ms_d * 1e-3) / 1e9
    res["decode"] = {"value": round(gbs, 1), "unit": "GB/s", "ms": round(ms_d, 4), "bytes": dec_bytes,
                     "frac": round(gbs / peaks["hbm_gbs"], 4), "peak": peaks["hbm_gbs"],
                     "workload": "64 seqs, ctx ~ U[512,32768] (seeded), 16-token pages, permuted pool, Hq32/Hkv8/D128",
                     "sum_ctx": int(ctx.sum())}
    del kp, vp
    torch.cuda.empty_cache()
    res["decode_long"] = measure_decode_long(torch, rlk, dv, peaks, flush, stream, args)
    res["rope"] = measure_rope(torch, rlk, dv, peaks, flush, stream, args)
    res["backward"] = measure_backward(torch, rlk, dv, peaks, flush, stream, args)
    res["chunked"] = measure_chunked(torch, rlk, dv, peaks, flush, stream, args)
    return res


def backward_workload(torch, rlk, dv):
    cfg = dict(synth.CFG_BACKWARD)
    prob = synth.prefill_problem(**cfg)
    q, k, v = dv.bf16_to_device(prob.q), dv.bf16_to_device(prob.k), dv.bf16_to_device(prob.v)
    T = q.shape[0]
    p = rlk.make_params(2, 32, 8, 128, 1, rlk.ZIGZAG, prob.scale)
    out = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
    lse = torch.empty((T, 32), dtype=torch.float32, device="cuda")
    rlk.rlk_attn_prefill(p, q, k, v, prob.cu_q, prob.cu_k, -1, out, None, lse)
    do = dv.bf16_to_device(synth.normal_bf16(cfg["seed"], synth.T_DOUT, prob.q.shape))
    dq = torch.empty((T, 32, 128), dtype=torch.float32, device="cuda")
    dk = torch.empty((T, 8, 128), dtype=torch.float32, device="cuda")
    dvv = torch.empty((T, 8, 128), dtype=torch.float32, device="cuda")
    ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_BACKWARD, prob.cu_q), dtype=torch.uint8,
                     device="cuda")
    flops = 2.5 * synth.prefill_flops(prob.cu_q, prob.cu_k, 32, 128)
    return prob, p, (q, k, v, out, do, lse, dq, dk, dvv, ws), flops


def measure_backward(torch, rlk, dv, peaks, flush, stream, args):
    """dQ/dK/dV of causal prefill, 2 x 4096 tokens, 32/8/128: algorithmic
    TFLOP/s = 2.5 x forward flops (five matmul-equivalents)."""
    prob, p, (q, k, v, out, do, lse, dq, dk, dvv, ws), flops = backward_workload(torch, rlk, dv)
    t = time_steps(torch, lambda: rlk.rlk_attn_backward(p, q, k, v, out, do, lse, prob.cu_q, -1, dq, dk, dvv, ws,
                                                         stream=stream),
                   args.steps, args.warmup, flush, stream)
    rlk.rlk_attn_check_device_error(stream)
    ms = float(np.mean(t))
    tf = flops / (ms * 1e-3) / 1e12
    return {"value": round(tf, 2), "unit": "TFLOP/s", "ms": round(ms, 4), "flops": flops,
            "frac": round(tf / peaks["bf16_tflops"], 4), "peak": peaks["bf16_tflops"],
            "workload": "2 x 4096 causal, Hq32/Hkv8/D128, dout ~ N(0,1) bf16; preprocess + dK/dV + dQ kernels"}


def measure_rope(torch, rlk, dv, peaks, flush, stream, args):
    """The RoPE pass over the varlen prefill workload's Q (32 heads) and K
    (8 heads), in place: 256 B read + 256 B written per (token, head) row."""
    cfg = synth.CFG_PREFILL
    cu = synth.cu_seqlens(cfg["lens"])
    t = int(cu[-1])
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    q = torch.randn((t, cfg["hq"], 128), generator=g, device="cuda").to(torch.bfloat16)
    k = torch.randn((t, cfg["hkv"], 128), generator=g, device="cuda").to(torch.bfloat16)
    max_pos = max(cfg["lens"])
    table = torch.from_numpy(rlk.rlk_attn_rope_table(1.0e6, max_pos)).cuda()
    pr = rlk.make_params(len(cfg["lens"]), cfg["hq"], cfg["hkv"])

    def step():
        rlk.rlk_attn_rope_qk(pr, q, q, k, k, cu, None, table, max_pos, stream=stream)
    ts = time_steps(torch, step, args.steps, args.warmup, flush, stream)
    # the same after a flush that leaves L2 clean: the 512 MB write leaves up
    # to 129 MB of dirty lines whose write-back a 182 MB pass otherwise pays
    reader = torch.zeros(256 * 1024 * 1024 // 4, dtype=torch.float32, device="cuda")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    for i in range(args.warmup + args.steps):
        flush.zero_()
        reader.sum()
        torch.cuda._sleep(400000)
        if i >= args.warmup:
            starts[i - args.warmup].record(stream)
        step()
        if i >= args.warmup:
            ends[i - args.warmup].record(stream)
    torch.cuda.synchronize()
    tc = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    del reader
    rlk.rlk_attn_check_device_error(stream)
    nbytes = t * (cfg["hq"] + cfg["hkv"]) * 512
    ms, msc = float(np.mean(ts)), float(np.mean(tc))
    gbs, gbsc = nbytes / (ms * 1e-3) / 1e9, nbytes / (msc * 1e-3) / 1e9
    return {"value": round(gbs, 1), "unit": "GB/s", "ms": round(ms, 4), "bytes": nbytes, "launches_per_step": 1,
            "frac": round(gbs / peaks["hbm_gbs"], 4), "peak": peaks["hbm_gbs"],
            "clean_l2": {"ms": round(msc, 4), "gbs": round(gbsc, 1), "frac": round(gbsc / peaks["hbm_gbs"], 4),
                         "flush": "512 MB write, then a 256 MB read (L2 left holding clean lines)"},
            "workload": "RoPE in place on the varlen prefill Q [8897,32,128] and K [8897,8,128] (BF16), one launch"}


def measure_prefill_rope(torch, rlk, peaks, prob, q, k, v, flush, stream, args, plain_ms):
    """The headline prefill with the queries' RoPE applied by the call
    (pre-RoPE q, post-RoPE k; whole sequences, so one pass rotates the
    queries into the output buffer and the fused kernel reads them there):
    against the plain prefill and against a RoPE pass into a separate
    buffer followed by the plain prefill."""
    rows = q.shape[0]
    max_pos = int(np.diff(prob.cu_k).max())
    table = torch.from_numpy(rlk.rlk_attn_rope_table(1.0e6, max_pos)).cuda()
    p = rlk.make_params(4, 32, 8, 128, 1, rlk.ZIGZAG, prob.scale)
    out = torch.empty((rows, 32, 128), dtype=torch.float32, device="cuda")
    outb = torch.empty((rows, 32, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows, 32), dtype=torch.float32, device="cuda")
    qr = torch.empty_like(q)
    pr = rlk.make_params(4, 32, 8)
    t_fused = time_steps(torch, lambda: rlk.rlk_attn_prefill_rope(p, q, k, v, prob.cu_q, prob.cu_k, -1, table, max_pos,
                                                                   out, outb, lse, stream=stream),
                         args.steps, args.warmup, flush, stream)

    def two_step():
        rlk.rlk_attn_rope(pr, q, qr, 32, prob.cu_q, None, table, max_pos, stream=stream)
        rlk.rlk_attn_prefill(p, qr, k, v, prob.cu_q, prob.cu_k, -1, out, outb, lse, stream=stream)
    t_two = time_steps(torch, two_step, args.steps, args.warmup, flush, stream)
    rlk.rlk_attn_check_device_error(stream)
    flops = synth.prefill_flops(prob.cu_q, prob.cu_k, 32, 128)
    ms, ms2 = float(np.mean(t_fused)), float(np.mean(t_two))
    return {"value": round(flops / (ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s", "ms": round(ms, 4),
            "vs_plain_prefill": round(ms / plain_ms, 4), "rope_pass_then_prefill_ms": round(ms2, 4),
            "workload": "the headline prefill with pre-RoPE queries, rotated by the call into the output buffer (RoPE theta 1e6)"}


def measure_decode_long(torch, rlk, dv, peaks, flush, stream, args, n=4, ctx_len=32768, split_k=(4, 8, 19)):
    """Few long sequences: n sequences of ctx_len tokens (n x 8 (sequence, KV
    head) items leave most SMs idle in a single pass), single-pass decode
    against the split decode with the library's automatic split_k and a few
    fixed ones; GB/s of the
    K+V bytes read (the split's state table traffic is counted as overhead,
    not work)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    ctx = np.full(n, ctx_len, np.int32)
    pages_per = (ctx + 15) // 16
    n_pages = int(pages_per.sum())
    perm = synth.rng(5, synth.T_PAGES).permutation(n_pages).astype(np.int32)
    pt = perm.reshape(n, -1).copy()
    kp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    vp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    qd = torch.randn((n, 32, 128), generator=g, device="cuda", dtype=torch.float32).to(torch.bfloat16)
    ptd = dv.i32_to_device(pt)
    pd = rlk.make_params(n, 32, 8, 128)
    o = torch.empty((n, 32, 128), dtype=torch.float32, device="cuda")
    ob = torch.empty((n, 32, 128), dtype=torch.bfloat16, device="cuda")
    lo = torch.empty((n, 32), dtype=torch.float32, device="cuda")
    ws = torch.empty(rlk.rlk_attn_workspace_size(pd, rlk.RLK_OP_DECODE_SPLIT, None, ctx), dtype=torch.uint8,
                     device="cuda")
    kv_bytes = int(ctx.astype(np.int64).sum()) * 8 * 128 * 2 * 2
    t1 = time_steps(torch, lambda: rlk.rlk_attn_decode_paged(pd, qd, kp, vp, n_pages, 16, ptd, pt.shape[1], ctx, o, ob,
                                                              lo, stream=stream), args.steps, args.warmup, flush, stream)
    split = {"auto_k": rlk.rlk_attn_decode_auto_split(pd, ctx, torch.cuda.get_device_properties(0).multi_processor_count)}
    for k in (0,) + tuple(split_k):
        ts = time_steps(torch, lambda: rlk.rlk_attn_decode_paged_splitk(pd, qd, kp, vp, n_pages, 16, ptd, pt.shape[1],
                                                                         ctx, k, o, ob, lo, ws, stream=stream),
                        args.steps, args.warmup, flush, stream)
        mss = float(np.mean(ts))
        split["auto" if k == 0 else str(k)] = {"ms": round(mss, 4), "gbs": round(kv_bytes / (mss * 1e-3) / 1e9, 1)}
    rlk.rlk_attn_check_device_error(stream)
    ms1 = float(np.mean(t1))
    return {"single_pass_gbs": round(kv_bytes / (ms1 * 1e-3) / 1e9, 1), "single_pass_ms": round(ms1, 4),
            "split": split, "kv_bytes": kv_bytes, "peak": peaks["hbm_gbs"],
            "workload": f"{n} seqs x {ctx_len} tokens, 16-token pages, Hq32/Hkv8/D128"}


def measure_chunked(torch, rlk, dv, peaks, flush, stream, args, chunk=2048):
    """Chunked-prefill replay (TP=2 shard: 2 x 8192 tokens, Hq16/Hkv4/D128):
    each sequence's queries in chunks of `chunk` tokens against the growing
    KV cache, one launch per chunk; algorithmic TFLOP/s of the causal
    attention the replay computes (the same flops as the full prefill)."""
    cfg = dict(synth.CFG_CHUNKED)
    prob = synth.prefill_problem(**cfg)
    q, k, v = dv.bf16_to_device(prob.q), dv.bf16_to_device(prob.k), dv.bf16_to_device(prob.v)
    rows = q.shape[0]
    out = torch.empty((rows, prob.hq, 128), dtype=torch.float32, device="cuda")
    outb = torch.empty((rows, prob.hq, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((rows, prob.hq), dtype=torch.float32, device="cuda")
    p1 = rlk.make_params(1, prob.hq, prob.hkv, prob.block, 1, rlk.ZIGZAG, prob.scale)
    calls = []
    for s_ in range(len(prob.cu_q) - 1):
        q0, q1, k0 = int(prob.cu_q[s_]), int(prob.cu_q[s_ + 1]), int(prob.cu_k[s_])
        for c0 in range(0, q1 - q0, chunk):
            c1 = min(c0 + chunk, q1 - q0)
            calls.append((q[q0 + c0:q0 + c1], k[k0:k0 + c1], v[k0:k0 + c1], [0, c1 - c0], [0, c1],
                          out[q0 + c0:q0 + c1], outb[q0 + c0:q0 + c1], lse[q0 + c0:q0 + c1]))

    def step():
        for (qq, kk, vv, cq, ck, oo, ob, ll) in calls:
            rlk.rlk_attn_prefill(p1, qq, kk, vv, cq, ck, -1, oo, ob, ll, stream=stream)

    t = time_steps(torch, step, args.steps, args.warmup, flush, stream)
    rlk.rlk_attn_check_device_error(stream)
    ms = float(np.mean(t))
    flops = synth.prefill_flops(prob.cu_q, prob.cu_k, prob.hq, prob.d)
    tf = flops / (ms * 1e-3) / 1e12
    return {"value": round(tf, 2), "unit": "TFLOP/s", "ms": round(ms, 4), "flops": flops, "chunk": chunk,
            "launches_per_step": len(calls), "frac": round(tf / peaks["bf16_tflops"], 4),
            "workload": "2 x 8192 (TP=2 shard, Hq16/Hkv4/D128), queries in chunks against the growing cache"}


def cpu_baseline(seconds_target):
    """The oracle (FP64 definition, OpenMP) on a bounded sample of the prefill
    workload's rows, in TFLOP/s of the rows it computed."""
    import oracle
    prob, _ = prefill_workload()
    oracle.build()
    rows = np.arange(0, prob.q.shape[0], 1, dtype=np.int64)
    # visible keys per row (bottom-right causal)
    vis = np.empty(len(rows), np.int64)
    for s in range(len(prob.cu_q) - 1):
        a, b = prob.cu_q[s], prob.cu_q[s + 1]
        vis[a:b] = np.arange(1, b - a + 1)
    # calibrate on a small sample, then size the sample for ~seconds_target
    rng = np.random.default_rng(0)
    cal = np.sort(rng.choice(rows, 64, replace=False))
    t0 = time.perf_counter()
    oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=cal)
    dt = time.perf_counter() - t0
    per_key = dt / max(1, vis[cal].sum())
    target_keys = seconds_target / per_key
    frac = min(1.0, target_keys / vis.sum())
    n = max(64, int(frac * len(rows)))
    sample = np.sort(rng.choice(rows, n, replace=False))
    t0 = time.perf_counter()
    oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=sample)
    dt = time.perf_counter() - t0
    flops = 4.0 * 128 * 32 * float(vis[sample].sum())
    return {"value": round(flops / dt / 1e12, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
            "kind": "oracle", "seconds": round(dt, 2),
            "sample": f"{n} of {len(rows)} query rows (all 32 heads) of the prefill workload, uniformly drawn, seed 0"}


def run_reference(args):
    """The oracle as the reference arm, on the host cores."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle
    oracle.build()
    prob, _ = prefill_workload()
    vis = np.empty(prob.q.shape[0], np.int64)
    for s in range(len(prob.cu_q) - 1):
        a, b = prob.cu_q[s], prob.cu_q[s + 1]
        vis[a:b] = np.arange(1, b - a + 1)
    rng = np.random.default_rng(1)
    n = args.reference_rows
    times, flops = [], []
    for i in range(args.warmup + args.steps):
        sample = np.sort(rng.choice(prob.q.shape[0], n, replace=False))
        t0 = time.perf_counter()
        oracle.attention_f64(prob.q, prob.k, prob.v, prob.cu_q, prob.cu_k, prob.scale, rows=sample)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            flops.append(4.0 * 128 * 32 * float(vis[sample].sum()))
    value = sum(flops) / sum(times) / 1e12
    ms = 1e3 * float(np.mean(times))
    sample_desc = f"{n} random query rows (all 32 heads) of the prefill workload per step"
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 0,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "sample": sample_desc},
            "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample_desc},
            "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_profile(args):
    """Run one entry point a few times without timing, for ncu captures:
    --profile prefill|states|merge|decode|decode-small|decode-long|rope|backward."""
    import torch
    import deterministic_context_attention_gb300 as rlk
    from deterministic_context_attention_gb300 import build as rbuild
    from deterministic_context_attention_gb300 import device as dv
    rbuild.build()
    rlk.load()
    stream = torch.cuda.current_stream()
    n = args.profile_iters
    if args.profile == "rope":
        # RoPE in place on the varlen prefill workload's Q and K, one launch
        cfg = synth.CFG_PREFILL
        cu = synth.cu_seqlens(cfg["lens"])
        t = int(cu[-1])
        q = dv.bf16_to_device(synth.normal_bf16(cfg["seed"], synth.T_Q, (t, cfg["hq"], 128)))
        k = dv.bf16_to_device(synth.normal_bf16(cfg["seed"], synth.T_K, (t, cfg["hkv"], 128)))
        max_pos = max(cfg["lens"])
        table = torch.from_numpy(rlk.rlk_attn_rope_table(1.0e6, max_pos)).cuda()
        pr = rlk.make_params(len(cfg["lens"]), cfg["hq"], cfg["hkv"])
        for _ in range(n):
            rlk.rlk_attn_rope_qk(pr, q, q, k, k, cu, None, table, max_pos, stream=stream)
    elif args.profile == "decode-long":
        # few long sequences: 4 x 32768 tokens, split decode with split_k 4
        g = torch.Generator(device="cuda")
        g.manual_seed(5)
        ctx = np.full(4, 32768, np.int32)
        n_pages = int(((ctx + 15) // 16).sum())
        pt = synth.rng(5, synth.T_PAGES).permutation(n_pages).astype(np.int32).reshape(4, -1).copy()
        kp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
        vp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
        qd = torch.randn((4, 32, 128), generator=g, device="cuda").to(torch.bfloat16)
        ptd = dv.i32_to_device(pt)
        pd = rlk.make_params(4, 32, 8, 128)
        o = torch.empty((4, 32, 128), dtype=torch.float32, device="cuda")
        ob = torch.empty((4, 32, 128), dtype=torch.bfloat16, device="cuda")
        l = torch.empty((4, 32), dtype=torch.float32, device="cuda")
        ws = torch.empty(rlk.rlk_attn_workspace_size(pd, rlk.RLK_OP_DECODE_SPLIT, None, ctx), dtype=torch.uint8,
                         device="cuda")
        for _ in range(n):
            rlk.rlk_attn_decode_paged_splitk(pd, qd, kp, vp, n_pages, 16, ptd, pt.shape[1], ctx, 4, o, ob, l, ws,
                                             stream=stream)
    elif args.profile == "backward":
        prob, p, (q, k, v, out, do, lse, dq, dk, dvv, ws), _ = backward_workload(torch, rlk, dv)
        for _ in range(n):
            rlk.rlk_attn_backward(p, q, k, v, out, do, lse, prob.cu_q, -1, dq, dk, dvv, ws, stream=stream)
    elif args.profile in ("decode", "decode-small"):
        # decode-small: the same shape with contexts up to 4096 tokens (about
        # 0.6 GB of pages, above L2) for captures that replay many passes
        g = torch.Generator(device="cuda")
        g.manual_seed(3)
        hi = 4097 if args.profile == "decode-small" else 32769
        ctx = synth.rng(3, synth.T_LENS).integers(512, hi, size=64).astype(np.int32)
        pages_per = (ctx + 15) // 16
        n_pages = int(pages_per.sum())
        perm = synth.rng(3, synth.T_PAGES).permutation(n_pages).astype(np.int32)
        pt = np.full((64, int(pages_per.max())), -1, np.int32)
        off = 0
        for s_ in range(64):
            pt[s_, :pages_per[s_]] = perm[off:off + pages_per[s_]]
            off += pages_per[s_]
        kp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
        vp = torch.randn((n_pages, 16, 8, 128), generator=g, device="cuda").to(torch.bfloat16)
        qd = torch.randn((64, 32, 128), generator=g, device="cuda").to(torch.bfloat16)
        ptd = dv.i32_to_device(pt)
        pd = rlk.make_params(64, 32, 8, 128)
        o = torch.empty((64, 32, 128), dtype=torch.float32, device="cuda")
        ob = torch.empty((64, 32, 128), dtype=torch.bfloat16, device="cuda")
        l = torch.empty((64, 32), dtype=torch.float32, device="cuda")
        for _ in range(n):
            rlk.rlk_attn_decode_paged(pd, qd, kp, vp, n_pages, 16, ptd, pt.shape[1], ctx, o, ob, l, stream=stream)
    else:
        prob, _ = prefill_workload()
        q, k, v = dv.bf16_to_device(prob.q), dv.bf16_to_device(prob.k), dv.bf16_to_device(prob.v)
        rows = q.shape[0]
        p = rlk.make_params(4, 32, 8, 128, 1, rlk.ZIGZAG, prob.scale)
        out = torch.empty((rows, 32, 128), dtype=torch.float32, device="cuda")
        outb = torch.empty((rows, 32, 128), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((rows, 32), dtype=torch.float32, device="cuda")
        if args.profile == "prefill":
            for _ in range(n):
                rlk.rlk_attn_prefill(p, q, k, v, prob.cu_q, prob.cu_k, -1, out, outb, lse, stream=stream)
        else:
            slabs, npairs = rlk.rlk_attn_plan_states(p, prob.cu_q, prob.cu_k, -1, 0)
            so = torch.empty((npairs, 128), dtype=torch.float32, device="cuda")
            sl = torch.empty((npairs,), dtype=torch.float32, device="cuda")
            ds = dv.slabs_to_device(slabs)
            ws = torch.empty(rlk.rlk_attn_workspace_size(p, rlk.RLK_OP_MERGE, prob.cu_q, prob.cu_k),
                             dtype=torch.uint8, device="cuda")
            for _ in range(n):
                rlk.rlk_attn_prefill_states(p, q, k, v, prob.cu_q, prob.cu_k, -1, 0, so, sl, stream=stream)
                if args.profile == "merge":
                    rlk.rlk_attn_merge_states(p, prob.cu_q, prob.cu_k, ds, len(slabs), so, sl, out, outb, lse, ws,
                                              stream=stream)
    torch.cuda.synchronize()
    rlk.rlk_attn_check_device_error(stream)
    print("profile run ok:", args.profile, n)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--reference-rows", type=int, default=512)
    ap.add_argument("--profile", default=None,
                    choices=["prefill", "states", "merge", "decode", "decode-small", "decode-long", "rope",
                             "backward"])
    ap.add_argument("--profile-iters", type=int, default=3)
    args = ap.parse_args()
    if args.profile:
        run_profile(args)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
