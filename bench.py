"""Prefill throughput of the clef-flash 32-layer hybrid decoder on GB300 (one JSON line).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload l16384|l512|b32x512]
                    [--impl clef|reference]

A step is one full prefill (embedding gather, 24 Gated DeltaNet + 8 gated full-attention layers,
final RMSNorm) of the workload's synthetic requests through clef_prefill_forward.  Default
workload: one request of 16,384 positions (the longest prefill; the 32-layer L=16384 target).
Weights are seeded random LUT-6 weights of the model's shapes; ids are uniform over the
248,320-token vocabulary.  Inputs (5.2 GB of packed weights per step) are far larger than L2.

With --gpus N (launched by torchrun, one rank per GPU) every rank runs its own replica on its
own requests: the path has no exchange step, so there is no collective on the data path
(weak scaling); the barrier and the max-over-ranks timing are the only communication.

The line's headline is --workload (default: one request of 16,384 positions); the metric's other
workloads (one request of 512 positions, 32 requests of 512 positions in one launch sequence)
are timed in the same run and reported under "workloads", each with its own step time, rooflines
and end-to-end number.

--impl reference times the oracle (plain C++ fp64 with OpenMP, CPU) as it stands, on a bounded
sample of the same workload extrapolated per layer, in the same metric and unit; rank 0 only.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "prefill tokens/s, 32-layer hybrid (L=512, L=16384); % of HBM/tensor roofline"
# DRAM bytes (read + written) per LUT-6 GEMM launch, averaged over the 128 launches of one
# 16,384-position prefill: ncu dram__bytes_read.sum + dram__bytes_write.sum of each of the eight
# launch shapes, captured in their decoder layers at 16,384 positions; no capture for the other
# workloads.
GEMM_DRAM_BYTES_PER_LAUNCH = {"l16384": 1016.8e6}

WORKLOADS = {
    "l16384": dict(B=1, L=16384, desc="32-layer hybrid prefill, 1 request x 16384 positions"),
    "l512": dict(B=1, L=512, desc="32-layer hybrid prefill, 1 request x 512 positions"),
    "b32x512": dict(B=32, L=512, desc="32-layer hybrid prefill, 32 independent requests x 512 positions"),
}


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=d["hbm_gbs"], tc_burst=d["bf16_tflops"], tc_sust=d["bf16_tflops_sustained"],
                    source="measured")
    return dict(hbm=6800.0, tc_burst=1900.0, tc_sust=1700.0, source="fallback")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"clef_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.remove(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def request_seed(rank):
    """Seed of the synthetic token ids of a rank's requests: every replica prefills its own."""
    return 1000 + rank


def slowest_rank_ms(ms, world, device=None):
    """The timed region's length on the slowest rank (max over ranks; the local value at N = 1)."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(B, L, steps, world, slowest_ms):
    """Whole-job throughput: the tokens all ranks prefilled over the slowest rank's time."""
    return B * L * steps * world / (slowest_ms / 1000.0)


# Algorithmic work of one prefill: every LUT-6 weight (and every fp16 a/b projection weight) is
# 2 flops per token, attention 4 * 256 * 16 * L(L+1)/2 per request and layer, the gated delta
# rule 6 d^2 per token and value head; padded or recomputed work is not counted.
LUT6_WEIGHTS = 6_912_212_992
AB_WEIGHTS = 24 * 2 * 32 * 4096          # the fp16 a/b projections of the GDN layers


def step_flops(B, L):
    gemm = 2.0 * (LUT6_WEIGHTS + AB_WEIGHTS) * B * L
    attn = 8 * 4.0 * 256 * 16 * L * (L + 1) / 2 * B
    gdn = 24 * 6.0 * 128 * 128 * 32 * B * L
    return gemm + attn + gdn


_ORACLE_INPUTS = {}


def oracle_rate(seed, ids_row, B, L, n1=64, n2=192, rows=8):
    """The oracle (C++, fp64) timed on this host's cores, extrapolated per layer to B requests of
    L positions.  A decoder layer's oracle time is a fixed part (dequantising its weights) plus a
    part linear in the positions, plus for an attention layer the softmax over all earlier keys,
    quadratic in L.  Timed: one GDN layer (layer 0) and one attention layer (layer 3) on the
    first n1 and on the first n2 positions of the request (the two give the fixed and the
    per-position parts), and the oracle's attention for the last `rows` query rows of a request
    of the full length L (16 query heads over L keys: the cost per (row, key) pair).  Returns
    (tokens/s for B x L, seconds of oracle time spent, description)."""
    import numpy as np

    import synth
    from oracle import _lib
    from oracle import layers as Lr
    from oracle import model as om

    spent = 0.0
    fit = {}
    for layer in (0, 3):
        key = ("w", seed, layer)
        if key not in _ORACLE_INPUTS:                  # drawn once per process, not timed
            _ORACLE_INPUTS[key] = synth.layer_weights(seed, layer)
        w = _ORACLE_INPUTS[key]
        t = {}
        for n in (n1, n2):
            x = synth.embedding_rows(seed, ids_row[:n]).astype(np.float64)
            t0 = time.perf_counter()
            om.decoder_layer(x, w, synth.is_attention_layer(layer))
            t[n] = time.perf_counter() - t0
            spent += t[n]
        per_pos = max(t[n2] - t[n1], 0.0) / (n2 - n1)
        fit[layer] = (t[n1] - n1 * per_pos, per_pos)
    r = min(rows, L)
    key = ("qkv", seed, L)
    if key not in _ORACLE_INPUTS:
        _ORACLE_INPUTS[key] = (synth.normal_f64(seed, "cpu.q", 0, (L, 16, 256)),
                               synth.normal_f64(seed, "cpu.k", 0, (L, 4, 256)),
                               synth.normal_f64(seed, "cpu.v", 0, (L, 4, 256)))
    q, k, v = _ORACLE_INPUTS[key]
    t0 = time.perf_counter()
    Lr.causal_attention(q, k, v, rows=(L - r, L))
    t_rows = time.perf_counter() - t0
    spent += t_rows
    pairs = sum(L - i for i in range(r))                    # keys seen by the last r rows
    per_pair = t_rows / pairs
    c_g, s_g = fit[0]
    c_a, s_a = fit[3]
    per_request = (24 * (c_g + L * s_g) + 8 * (c_a + L * s_a + per_pair * L * (L + 1) / 2))
    total = B * per_request
    desc = (f"oracle (C++ fp64, {_lib.lib().orc_num_threads()} threads) extrapolated per layer to "
            f"{B} x {L} positions: GDN layer 0 and attention layer 3 timed on the first {n1} and "
            f"{n2} positions (fixed + per-position cost), the causal softmax timed on the last "
            f"{r} query rows of a {L}-position request (its quadratic term at {L} keys); "
            f"24 GDN + 8 attention layers")
    return B * L / total, spent, desc


def run_reference(args, wl):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import synth
    from oracle import _lib
    ids = synth.token_ids(request_seed(0), wl["B"], wl["L"])
    vals = []
    for _ in range(args.warmup):
        oracle_rate(0, ids[0], wl["B"], wl["L"], n1=32, n2=64, rows=4)
    t_all = 0.0
    desc = ""
    for _ in range(args.steps):
        v, t, desc = oracle_rate(0, ids[0], wl["B"], wl["L"], n1=32, n2=64, rows=4)
        vals.append(v)
        t_all += t
    value = statistics.median(vals)
    cores = int(_lib.lib().orc_num_threads())
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * t_all / max(1, args.steps),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": wl["desc"], "global_batch": wl["B"], "seq_len": wl["L"]},
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": desc},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def measure(model, ids_np, steps, warmup, world, dev, lib_trace=True):
    """Time `steps` prefills of the requests ids_np [B, L] (device-resident inputs), then the same
    steps with the library's per-launch trace, then end to end from pinned host memory."""
    import torch

    import full_attention_prefill_gb300 as clef

    B, L = ids_np.shape
    ids = torch.from_numpy(ids_np).to(dev)
    out = torch.empty((B, L, 4096), dtype=torch.float16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()

    for _ in range(warmup):
        model.forward(ids, out=out)
    clef.sync_status()

    # ---- timed region: device-resident inputs, no instrumentation
    clocks = ClockSampler(dev.index)
    clocks.start()
    barrier()
    torch.cuda.synchronize(dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    ev[0].record(stream)
    for i in range(steps):
        model.forward(ids, out=out)
        ev[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier()
    clk = clocks.stop()
    clef.sync_status()
    step_ms = [ev[i].elapsed_time(ev[i + 1]) for i in range(steps)]
    total_ms = slowest_rank_ms(ev[0].elapsed_time(ev[-1]), world, dev)

    # ---- the same steps again with the library's trace on (CUDA events around every launch,
    # on the launch stream): per-kernel times for the roofline and the breakdown
    lib = clef.lib()
    lib.clef_trace_begin.restype = ctypes.c_int
    lib.clef_trace_end.argtypes = [ctypes.POINTER(TraceEntry), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    torch.cuda.synchronize(dev)
    lib.clef_trace_begin()
    tv0, tv1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    tv0.record(stream)
    for i in range(steps):
        model.forward(ids, out=out)
    tv1.record(stream)
    torch.cuda.synchronize(dev)
    traced_ms = tv0.elapsed_time(tv1) / steps
    entries = (TraceEntry * 32)()
    n = ctypes.c_int32(0)
    rc = lib.clef_trace_end(entries, 32, ctypes.byref(n))
    clef.sync_status()
    trace = {}
    if rc == 0:
        for i in range(n.value):
            e = entries[i]
            trace[e.name.decode()] = dict(launches=e.launches, ms=e.ms, flops=e.flops, bytes=e.bytes)

    # ---- end to end through the public API: pinned host ids in, pinned host hidden out
    ids_host = torch.from_numpy(ids_np).pin_memory()
    out_host = torch.empty((B, L, 4096), dtype=torch.float16).pin_memory()
    ids_dev = torch.empty_like(ids)
    for _ in range(max(1, warmup // 2)):
        ids_dev.copy_(ids_host, non_blocking=True)
        model.forward(ids_dev, out=out)
        out_host.copy_(out, non_blocking=True)
    torch.cuda.synchronize(dev)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        ids_dev.copy_(ids_host, non_blocking=True)
        model.forward(ids_dev, out=out)
        out_host.copy_(out, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    e2e_ms = slowest_rank_ms(e0.elapsed_time(e1), world, dev)
    return dict(B=B, L=L, total_ms=total_ms, step_ms=step_ms, clocks=clk, trace=trace,
                traced_ms=traced_ms, e2e_ms=e2e_ms, h2d=int(ids_host.numel() * 4),
                d2h=int(out_host.numel() * 2))


def summarize(r, steps, world, pk, traffic=None):
    """The metric's numbers of one measured workload."""
    B, L = r["B"], r["L"]
    value = job_tokens_per_s(B, L, steps, world, r["total_ms"])
    ms = r["total_ms"] / steps
    g = r["trace"].get("lut6_gemm")
    gemm = None
    if g and g["ms"] > 0:
        per_launch_flops = g["flops"] / g["launches"]
        avg_ms = g["ms"] / g["launches"]
        achieved = per_launch_flops / (avg_ms / 1000.0) / 1e12
        gemm = {"bound": "tensor", "achieved": achieved, "peak": pk["tc_sust"], "unit": "TFLOP/s",
                "frac": achieved / pk["tc_sust"], "traffic": traffic, "kernel": "lut6_gemm",
                "peak_kind": f"bf16 dense sustained ({pk['source']}), fp16 same nominal rate",
                "algorithmic_flops_per_launch": per_launch_flops, "avg_launch_ms": avg_ms}
    sf = step_flops(B, L)
    whole = {"bound": "tensor", "achieved": sf / (ms / 1000.0) / 1e12, "peak": pk["tc_sust"],
             "unit": "TFLOP/s", "frac": sf / (ms / 1000.0) / 1e12 / pk["tc_sust"],
             "algorithmic_flops_per_step": sf,
             "what": "whole prefill: LUT-6 GEMMs + a/b projections + attention + gated delta rule"}
    return dict(value=value, ms_per_step=ms, gemm=gemm, whole=whole,
                e2e={"value": job_tokens_per_s(B, L, steps, world, r["e2e_ms"]), "unit": "tokens/s",
                     "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"]},
                launches=int(sum(t["launches"] for t in r["trace"].values()) / steps) if r["trace"] else None)


def run_clef(args, wl):
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    import synth
    from full_attention_prefill_gb300.model import synth_model

    model = synth_model(0, 32, device=dev)
    pk = peaks()
    # the headline workload, then the metric's other workloads in the same run
    names = [args.workload] + [w for w in ("l512", "b32x512", "l16384") if w != args.workload
                               and not args.only_headline]
    results = {}
    for name in names:
        w = WORKLOADS[name]
        ids_np = synth.token_ids(request_seed(rank), w["B"], w["L"])   # each rank: its own requests
        results[name] = measure(model, ids_np, args.steps, args.warmup, world, dev)

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    head = results[args.workload]
    hs = summarize(head, args.steps, world, pk, GEMM_DRAM_BYTES_PER_LAUNCH.get(args.workload))
    ids0 = synth.token_ids(request_seed(0), 1, wl["L"])[0]
    cpu_v, cpu_s, cpu_desc = oracle_rate(0, ids0, wl["B"], wl["L"])
    trace = head["trace"]
    step_total = sum(t["ms"] for t in trace.values()) / args.steps if trace else None
    others = {}
    for name in names[1:]:
        r = results[name]
        sm = summarize(r, args.steps, world, pk, GEMM_DRAM_BYTES_PER_LAUNCH.get(name))
        others[name] = {
            "workload": WORKLOADS[name]["desc"], "global_batch": r["B"] * world, "seq_len": r["L"],
            "value": sm["value"], "unit": "tokens/s", "ms_per_step": sm["ms_per_step"],
            "step_ms": {"median": statistics.median(r["step_ms"]), "min": min(r["step_ms"]),
                        "max": max(r["step_ms"])},
            "roofline": sm["gemm"], "roofline_whole_step": sm["whole"], "e2e": sm["e2e"],
            "gpu_launches_per_step": sm["launches"], "clocks": r["clocks"],
            "kernels_ms_per_step": {k: round(v["ms"] / args.steps, 3)
                                    for k, v in sorted(r["trace"].items(), key=lambda kv: -kv[1]["ms"])},
            "traced_ms_per_step": r["traced_ms"],
        }
    line = {
        "metric": METRIC, "value": hs["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": hs["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp16 activations, fp32 accumulate, LUT-6 weights",
        "data": "synthetic (seeded random LUT-6 weights and token ids)",
        "config": {"workload": wl["desc"], "global_batch": wl["B"] * world, "seq_len": wl["L"], "layers": 32,
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU",
                   "l2": "inputs larger than L2 (5.2 GB of packed weights streamed per step)"},
        "roofline": hs["gemm"],
        "roofline_whole_step": hs["whole"],
        "cpu_baseline": {"value": cpu_v, "unit": "tokens/s", "cores": int(__import__("oracle")._lib.lib().orc_num_threads()),
                         "kind": "oracle", "sample": cpu_desc, "oracle_seconds": cpu_s},
        "e2e": hs["e2e"],
        "gpu_launches": int(sum(t["launches"] for t in trace.values())) if trace else None,
        "clocks": head["clocks"],
        "step_ms": {"median": statistics.median(head["step_ms"]), "min": min(head["step_ms"]),
                    "max": max(head["step_ms"])},
        "kernels_ms_per_step": {k: round(v["ms"] / args.steps, 3) for k, v in sorted(trace.items(), key=lambda kv: -kv[1]["ms"])},
        "kernel_time_sum_ms_per_step": step_total,
        "traced_ms_per_step": head["traced_ms"],
        "kernel_times": "per-launch CUDA events on the launch stream, in a pass of the same steps "
                        "right after the timed region (the timed region runs without them)",
        "workloads": others,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


import ctypes  # noqa: E402


class TraceEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int64), ("ms", ctypes.c_double),
                ("flops", ctypes.c_double), ("bytes", ctypes.c_double)]


def run_micro(args):
    """One kernel entry point in a loop (CUDA events), for profiling and tuning.

    gemm: clef_lut6_gemm at M x N x K (fp16 out); attn: clef_gqa_attn_prefill at L (gated);
    gdn: clef_gdn_prefill at L; layer: clef_decoder_layer of layer --layer at L (the residual
    copy-in is part of each iteration); chunk: one request of L positions as calls of --chunk
    positions through clef_prefill_forward_chunk (zeroing the state is part of each iteration);
    quantize: clef_lut6_quantize of an N x K fp16 weight; image: a prefill of L positions with a
    14 x 14 picture block through clef_prefill_forward_image.  Prints one JSON line with the
    per-kernel times of the library's trace; not the headline metric.
    """
    import numpy as np
    import torch

    import full_attention_prefill_gb300 as clef
    import synth

    dev = torch.device("cuda", 0)
    pk = peaks()
    extra_fn = None
    if args.micro == "gemm":
        M, N, K = args.m, args.n, args.k
        x = torch.from_numpy(synth.normal_f16(0, "micro.x", 0, (M, K))).to(dev)
        packed, lut = synth.lut6_weight(0, "micro.w", 0, N, K)
        p, l = torch.from_numpy(packed).to(dev), torch.from_numpy(lut).to(dev)
        y = torch.empty((M, N), dtype=torch.float16, device=dev)
        if args.canonical:
            # the card's packing through clef_lut6_gemm_canonical (tiled into a workspace first)
            fn = lambda: clef.lut6_gemm(x, p, l, out=y)  # noqa: E731
        else:
            p = clef.lut6_tile(p, K)
            fn = lambda: clef.lut6_gemm(x, p, l, out=y, tiled=True)  # noqa: E731
        flops, desc = 2.0 * M * N * K, f"lut6_gemm M={M} N={N} K={K}" + (" canonical" if args.canonical else "")
    elif args.micro == "attn":
        L = args.L
        q = torch.from_numpy(synth.normal_f16(0, "q", 0, (1, L, 16, 256))).to(dev)
        k = torch.from_numpy(synth.normal_f16(0, "k", 0, (1, L, 4, 256))).to(dev)
        v = torch.from_numpy(synth.normal_f16(0, "v", 0, (1, L, 4, 256))).to(dev)
        g = torch.from_numpy(synth.normal_f16(0, "g", 0, (1, L, 16, 256))).to(dev)
        fn = lambda: clef.gqa_attn_prefill(q, k, v, g)  # noqa: E731
        flops, desc = 4.0 * 256 * 16 * L * (L + 1) / 2, f"gqa_attn L={L}"
    elif args.micro == "chunk":
        # one request of --L positions prefilled as calls of --chunk positions on a carried state
        from full_attention_prefill_gb300.model import PrefillState, synth_model
        L, C = args.L, args.chunk
        model = synth_model(0, 32, device=dev)
        ids = torch.from_numpy(synth.token_ids(1000, 1, L)).to(dev)
        calls = [ids[:, p:p + C].contiguous() for p in range(0, L, C)]
        st_box = []

        def fn():
            st = PrefillState(model, 1, L, dev)
            st_box[:] = [st]
            for c in calls:
                model.forward_chunk(c, st)
        flops, desc = 0.0, f"chunked prefill L={L} in calls of {C}"
        extra_fn = lambda ms: {"tokens_per_s": L / (ms / 1000.0), "ms_per_call": ms / len(calls)}  # noqa: E731
    elif args.micro == "image":
        # one request of --L positions holding a 14 x 14 picture block (196 tokens, the pages'
        # 448-pixel tile) at index 37, through clef_prefill_forward_image (M-RoPE rotary)
        from full_attention_prefill_gb300.model import synth_model
        L, grid = args.L, (14, 14)
        model = synth_model(0, 32, device=dev)
        ids = torch.from_numpy(synth.token_ids(1000, 1, L)).to(dev)
        rows = torch.from_numpy(synth.normal_f16(0, "micro.image", -1, (1, 196, 4096), 0.0, 0.05)).to(dev)
        out = torch.empty((1, L, 4096), dtype=torch.float16, device=dev)
        fn = lambda: model.forward_image(ids, rows, 37, grid, out=out)  # noqa: E731
        flops, desc = 0.0, f"picture prefill L={L}, 14x14 block at 37"
        extra_fn = lambda ms: {"tokens_per_s": L / (ms / 1000.0)}  # noqa: E731
    elif args.micro == "quantize":
        # LUT-6 quantisation of one fp16 weight [--n, --k] (default: the MLP down projection)
        N, K = args.n, args.k
        w = torch.from_numpy(synth.normal_f16(0, "micro.qw", 0, (N, K), std=0.02)).to(dev)
        fn = lambda: clef.lut6_quantize(w)  # noqa: E731
        flops, desc = 0.0, f"lut6_quantize N={N} K={K}"
        extra_fn = lambda ms: {"weights_per_s": N * K / (ms / 1000.0),  # noqa: E731
                               "groups_per_s": N / 16 / (ms / 1000.0),
                               "weight_GB_per_s": 2.0 * N * K / (ms * 1e6)}
    elif args.micro == "layer":
        # one decoder layer (GDN for --layer 0, attention for --layer 3) on an fp32 residual
        from full_attention_prefill_gb300.model import DeviceLayer, DeviceModel
        L = args.L
        layer = DeviceLayer(synth.layer_weights(0, args.layer), DeviceModel.kind_of(args.layer), dev)
        x0 = torch.from_numpy(synth.normal_f32(0, "micro.x", 0, (1, L, 4096))).to(dev)
        x = x0.clone()
        ws = torch.empty(clef.prefill_workspace_size(1, L), dtype=torch.uint8, device=dev)

        def fn():
            x.copy_(x0)
            clef.decoder_layer(layer, x, workspace=ws)
        flops, desc = 0.0, f"decoder_layer {args.layer} L={L}"
    else:
        L = args.L
        q = torch.from_numpy(synth.normal_f16(0, "q", 0, (1, L, 16, 128))).to(dev)
        k = torch.from_numpy(synth.normal_f16(0, "k", 0, (1, L, 16, 128))).to(dev)
        q = q / q.float().norm(dim=-1, keepdim=True).half()
        k = k / k.float().norm(dim=-1, keepdim=True).half()
        v = torch.from_numpy(synth.normal_f16(0, "v", 0, (1, L, 32, 128))).to(dev)
        a = torch.full((1, L, 32), 0.92, dtype=torch.float32, device=dev)
        b = torch.full((1, L, 32), 0.5, dtype=torch.float32, device=dev)
        fn = lambda: clef.gdn_prefill(q, k, v, a, b)  # noqa: E731
        flops, desc = 6.0 * 128 * 128 * 32 * L, f"gdn_scan L={L}"
    for _ in range(args.warmup):
        fn()
    clef.sync_status()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    lib = clef.lib()
    lib.clef_trace_begin()
    e0.record()
    for _ in range(args.steps):
        fn()
    e1.record()
    torch.cuda.synchronize()
    entries = (TraceEntry * 32)()
    n = ctypes.c_int32(0)
    lib.clef_trace_end.argtypes = [ctypes.POINTER(TraceEntry), ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)]
    rc = lib.clef_trace_end(entries, 32, ctypes.byref(n))
    clef.sync_status()
    ms = e0.elapsed_time(e1) / args.steps
    kernels = {}
    if rc == 0:
        for i in range(n.value):
            e = entries[i]
            kernels[e.name.decode()] = {"ms": round(e.ms / args.steps, 4),
                                        "GB/s": round(e.bytes / (e.ms * 1e6), 1) if e.ms > 0 else None}
        if flops == 0.0:
            flops = sum(entries[i].flops for i in range(n.value)) / args.steps
    line = {"micro": desc, "ms": ms, "kernels": kernels}
    if flops > 0:
        line.update(tflops=flops / ms / 1e9, frac_of_sustained=flops / ms / 1e9 / pk["tc_sust"])
    if extra_fn is not None:
        line.update(extra_fn(ms))
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--micro", choices=["gemm", "attn", "gdn", "layer", "chunk", "quantize", "image"], default=None)
    ap.add_argument("--chunk", type=int, default=64)
    ap.add_argument("--canonical", action="store_true",
                    help="--micro gemm: pass the card's packing (clef_lut6_gemm_canonical)")
    ap.add_argument("--layer", type=int, default=0)
    ap.add_argument("--m", type=int, default=4096)
    ap.add_argument("--n", type=int, default=24576)
    ap.add_argument("--k", type=int, default=4096)
    ap.add_argument("--L", type=int, default=4096)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["clef", "reference"], default="clef")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default="l16384")
    ap.add_argument("--only-headline", action="store_true",
                    help="time only --workload (the line then has no other workloads)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    wl = WORKLOADS[args.workload]
    if args.micro:
        run_micro(args)
    elif args.impl == "reference":
        run_reference(args, wl)
    else:
        run_clef(args, wl)


if __name__ == "__main__":
    main()
