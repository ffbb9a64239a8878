"""Benchmark of the MoE layer-step hot path on B300.

Default workload (the one the headline metric is quoted on): decode of one
token through 30 stacked MoE layers of the Gemma-4-26B-A4B block shape
(d_model 2816, 128 experts of inner size 704, top-8, shared expert 2112,
affine 4-bit g64 experts, 8-bit router), every expert resident in HBM.  One
step = one token through all 30 layers = one persistent kernel launch.

Prints one JSON line.  `--impl reference` times the plain CPU oracle on the
host cores on a bounded sample of the same workload instead.

Multi-GPU: the path does not shard (one GPU per model replica), so under
torchrun each rank runs an independent replica and `value` sums the tokens of
all ranks over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-layer tokens/s; expert-weight HBM GB/s as % of B300 peak (decode/prefill)"


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return d["hbm_gbs"], d["bf16_tflops"], "measured"
    except Exception:
        return 6400.0, 1800.0, "fallback"


def job_throughput(seconds: float, units_per_rank: float, world: int, device=None) -> float:
    """Whole-job throughput of independent replicas: every rank processed
    units_per_rank units; the job took as long as its slowest rank (max over
    ranks with a collective when world > 1)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return units_per_rank * world / float(t.item())


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", "moe_clocks_%d_%d.csv" % (os.getpid(), gpu_index))

    def start(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.f,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.unlink(self.path)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "samples": len(sm),
                "reasons": sorted(reasons)}


# DRAM traffic (read + write) of one 4-layer decode_kernel launch from the
# `--set full` capture summarised in profiles/decode_kernel_gemma30.md, and
# a hash of the kernel's sources when it was taken.  Reported, scaled to the
# launch's layers by the algorithmic bytes, only while the sources match.
DECODE_CAPTURE = {"sources_sha16": "87927194c7970c40", "traffic_bytes": 149384192 + 3215104,
                  "algo_bytes": 148729856}
DECODE_SOURCES = ["decode.cu", "qdot.cuh", "ptx.cuh", "internal.h"]


def decode_traffic(algo_bytes: int):
    import hashlib
    h = hashlib.sha256()
    try:
        for f in DECODE_SOURCES:
            with open(os.path.join(ROOT, "expert_ffn_streaming_bit_b300", "csrc", f), "rb") as fh:
                h.update(fh.read())
    except OSError:
        return None
    if h.hexdigest()[:16] != DECODE_CAPTURE["sources_sha16"]:
        return None
    return DECODE_CAPTURE["traffic_bytes"] * algo_bytes / DECODE_CAPTURE["algo_bytes"]


def decode_bytes_per_token(shape) -> int:
    """Algorithmic weight bytes one token reads through all layers (canonical sizes)."""
    return shape.n_layers * shape.decode_layer_bytes()


def make_layers(shape, workload, n_layers, device):
    import synth
    import torch
    out = []
    for l in range(n_layers):
        L = synth.make_layer(shape, workload, l, device=device)
        out.append(synth.layer_to(L, "cpu"))
        del L
    if device == "cuda":
        torch.cuda.empty_cache()
    return out


def decode_config(L: int, world: int) -> dict:
    """`config` of the decode line; the reference arm prints the same one."""
    return {"workload": "decode: %d stacked MoE layers, d_model 2816, 128 experts x 704, "
                        "top-8, shared 2112, 4-bit g64 experts, 8-bit router, T=1, all "
                        "experts resident in HBM" % L,
            "layers": L, "tokens_per_step": 1,
            "l2": "inputs larger than L2: 1.12 GB of expert weights read per token, "
                  "64 distinct tokens cycled",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def cpu_baseline_decode(shape, layers, L, budget_s: float) -> dict:
    """The oracle as it stands, one token through the stack, timed on the host
    at all cores and at one core (each a bounded sample of layers)."""
    import oracle
    import synth
    x0 = synth.make_tokens(shape, "decode", 1, index=3000)
    all_cores = oracle.set_threads(os.cpu_count() or 1)
    dt, n = oracle_sample(shape, layers, x0, budget_s)
    one = oracle.set_threads(1)
    dt1, n1 = oracle_sample(shape, layers, x0, budget_s)
    oracle.set_threads(all_cores)
    return {"value": 1.0 / (dt / n * L), "unit": "tokens/s", "cores": all_cores,
            "kind": "oracle",
            "sample": "one token through %d of the %d layers (%.1f s), scaled to %d layers"
                      % (n, L, dt, L),
            "one_core": {"value": 1.0 / (dt1 / n1 * L), "unit": "tokens/s", "cores": one,
                         "sample": "one token through %d of the %d layers (%.1f s), scaled "
                                   "to %d layers" % (n1, L, dt1, L)}}


def oracle_sample(shape, layers, x_cpu, budget_s: float):
    """Time the oracle on one token through as many layers as fit the budget."""
    import oracle
    t0 = time.perf_counter()
    n = 0
    x = x_cpu
    import torch
    while n < len(layers):
        ref = oracle.moe_layer(oracle.LayerView(shape, layers[n]), x, prenorm=True)
        y = torch.tensor(ref["y"], dtype=torch.float32)
        x = (x.float() + y).to(torch.bfloat16)
        n += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return dt, n


def run_ours(args):
    import torch
    import torch.distributed as dist
    import synth
    import expert_ffn_streaming_bit_b300 as moe

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    shape = synth.GEMMA
    L = args.layers or shape.n_layers
    layers = make_layers(shape, "decode", L, "cuda")
    # room for a 32-token batch (the batched-decode sub-record); single tokens
    # run the same decode kernel either way
    h = moe.moe_create(shape, layers, max_tokens=32)
    info = moe.moe_get_info(h)
    P = 64
    xs = synth.make_tokens(shape, "decode", P, index=1000 + rank).cuda()
    xrows = [xs[i:i + 1] for i in range(P)]
    ys = [torch.empty_like(xrows[0]) for _ in range(2)]
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        moe.moe_forward_stack(h, xrows[i % P], ys[i % 2], L)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    t_start.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        moe.moe_forward_stack(h, xrows[i % P], ys[i % 2], L)
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end)
    launch_ms = float(np.mean([s.elapsed_time(e) for s, e in zip(starts, ends)]))
    value = job_throughput(ms / 1e3, args.steps, world, device="cuda")
    ms_max = args.steps * world / value * 1e3
    # end to end through the host-I/O entry point: H2D of x, stack, D2H of y, per step
    xh = synth.make_tokens(shape, "decode", P, index=2000 + rank).view(torch.int16).numpy().view(np.uint16)
    yh = np.empty((1, shape.d_model), np.uint16)
    for i in range(min(args.warmup, 10)):
        moe.moe_forward_stack_host(h, xh[i % P:i % P + 1], yh, L)
    n_e2e = max(200, min(args.steps, 2000))
    te0 = time.perf_counter()
    for i in range(n_e2e):
        moe.moe_forward_stack_host(h, xh[i % P:i % P + 1], yh, L)
    te = time.perf_counter() - te0
    e2e_value = job_throughput(te, n_e2e, world, device="cuda")
    hbm, bf16, src = peaks()
    sub = synth.MoEShape(shape.name, shape.d_model, shape.n_experts, shape.d_expert, shape.top_k,
                         shape.d_shared, shape.group, L)
    algo = decode_bytes_per_token(sub)
    achieved = algo / (launch_ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_max / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "u4 x s16 -> s32 (dp2a) per 32-column chunk, f32 scale and sum",
        "data": "synthetic (seeded N(0,0.02) weights quantised to affine 4-bit g64; N(0,1) bf16 tokens)",
        "config": decode_config(L, world),
        "expert_weight_gbs": algo * value / world / 1e9,
        "hbm_frac_of_measured": algo * value / world / 1e9 / hbm,
        "hbm_frac_of_8tbs": algo * value / world / 1e9 / 8000.0,
        "roofline": {"bound": "hbm", "kernel": "decode_kernel", "achieved": achieved,
                     "peak": hbm, "peak_source": src, "unit": "GB/s", "frac": achieved / hbm,
                     "bytes_per_launch": algo, "avg_launch_ms": launch_ms,
                     "traffic": decode_traffic(algo),
                     "traffic_source": "ncu dram__bytes_read.sum + dram__bytes_write.sum of a "
                                       "4-layer launch, scaled by the algorithmic bytes"},
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 2 * shape.d_model,
                "d2h_bytes_per_step": 2 * shape.d_model, "api": "moe_forward_stack_host"},
        "gpu_launches": args.steps,
        "clocks": clk,
        "device": {"name": torch.cuda.get_device_name(local), "weight_bytes": info["device_weight_bytes"]},
    }
    if rank == 0 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_decode(shape, layers, L, args.cpu_budget)
    del layers
    if rank == 0 and not args.no_sub_records:
        # the full decode layer step on the same MoE handle: attention at a
        # 4096-token context, then the router and experts, for every layer
        layer_step = compact(measure_layer_step(args, h, L, context=4096, steps=50, warmup=5))
        batched = compact(measure_batched(args, h, L, 32, steps=20, warmup=3))
    moe.moe_destroy(h)
    torch.cuda.empty_cache()
    if rank == 0 and not args.no_sub_records:
        # the other workloads, timed in the same run on fewer steps
        line["sub_records"] = {
            "decode_layer_step_ctx4096": layer_step,
            "batched_decode_32": batched,
            "prefill_4096": compact(measure_prefill(args, steps=3, warmup=3)),
            "chunked_128": compact(measure_chunked(args, steps=2, warmup=3)),
            "streaming_pinned_4l": compact(measure_streaming(args, 32, 3, 4, None, False)),
            "streaming_store_4l": compact(measure_streaming(args, 32, 3, 4, args.store or "/tmp",
                                                            False)),
        }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def measure_layer_step(args, h, L, context, steps, warmup):
    """Full decode layer steps: for each of the L layers, decode attention
    (the Gemma-shape reading: 16 query heads over 8 kv heads of 256; every
    sixth layer full attention, the others a 1024-token window) at a context
    of `context` earlier tokens, then the router and the experts of the MoE
    handle h on the attention output (moe_decode_step).  The KV caches are
    filled first by attention steps over seeded tokens."""
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    ash = synth.GEMMA_ATTN
    alayers = []
    for l in range(L):
        A = synth.make_attn_layer(ash, "decode", l, device="cuda")
        alayers.append({k: v.to("cpu") for k, v in A.items()})
        del A
    torch.cuda.empty_cache()
    a = moe.moe_attn_create(ash, alayers)
    del alayers
    n = context + warmup + steps
    xs = synth.make_tokens(synth.GEMMA, "decode", 256, index=5000).cuda()
    y = torch.empty_like(xs[0:1])
    for p in range(context):                      # fill the caches
        for l in range(L):
            moe.moe_attn_forward(a, l, xs[p % 256:p % 256 + 1], p, y)
    torch.cuda.synchronize()
    for p in range(context, context + warmup):
        moe.moe_decode_step(a, h, xs[p % 256:p % 256 + 1], p, y, L)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for p in range(context + warmup, n):
        moe.moe_decode_step(a, h, xs[p % 256:p % 256 + 1], p, y, L)
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / steps
    hbm, bf16, src = peaks()
    kv_pos = sum(min(context + warmup + steps // 2, ash.window) if ash.sliding[l]
                 else context + warmup + steps // 2 for l in range(L))
    kv_bytes = kv_pos * ash.n_kv_heads * ash.head_dim * 2 * 2
    moe_bytes = L * synth.GEMMA.decode_layer_bytes()
    attn_bytes = L * ash.attn_weight_bytes()
    total = moe_bytes + attn_bytes + kv_bytes
    gbs = total / (ms / 1e3) / 1e9
    line = {
        "value": 1e3 / ms, "unit": "tokens/s", "ms_per_step": ms, "steps": steps, "warmup": warmup,
        "config": {"workload": "decode layer step: %d layers of attention (16 x 256 query heads, "
                               "8 kv heads, 1024-token window on 5 of 6 layers, full on every "
                               "sixth) at a %d-token context, then the MoE layer (128 experts, "
                               "top-8, shared 2112), T=1" % (L, context),
                   "layers": L, "context": context, "tokens_per_step": 1},
        "bytes_per_token": {"moe_weights": moe_bytes, "attention_weights": attn_bytes,
                            "kv_cache": kv_bytes},
        "roofline": {"bound": "hbm", "kernel": "whole layer step (attention + MoE)",
                     "achieved": gbs, "peak": hbm, "peak_source": src, "unit": "GB/s",
                     "frac": gbs / hbm, "traffic": None},
        "gpu_launches": 6 * L * steps,
        "clocks": clk,
        "dtype": "u4 x s16 -> s32 (dp2a) projections and experts; f16 KV, f32 softmax",
    }
    moe.moe_attn_destroy(a)
    torch.cuda.empty_cache()
    return line


def run_layer_step(args):
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    import torch
    torch.cuda.set_device(0)
    L = args.layers or 30
    layers = make_layers(synth.GEMMA, "decode", L, "cuda")
    h = moe.moe_create(synth.GEMMA, layers, max_tokens=1)
    del layers
    print(json.dumps(measure_layer_step(args, h, L, args.context, args.steps, args.warmup)),
          flush=True)


def gemm_flops_per_layer(shape, T):
    """Algorithmic FLOPs of the expert GEMMs of one layer for T tokens (routed
    gate/up + down over T*k rows, shared gate/up + down over T rows)."""
    D, I, S, k = shape.d_model, shape.d_expert, shape.d_shared, shape.top_k
    return 2 * T * k * (2 * I * D + D * I) + 2 * T * (2 * S * D + D * S)


def compact(line: dict) -> dict:
    """A workload's line without the keys the headline line already carries."""
    keep = ("value", "unit", "ms_per_step", "steps", "warmup", "config", "roofline",
            "whole_layer", "phase_ms_per_layer", "phase_ms_per_chunk_layer",
            "touched_weight_bytes_per_step", "bytes_per_token", "hit_rate", "misses_per_layer_step",
            "h2d_gbs", "h2d_link_gbs", "store", "overlap", "path", "e2e", "clocks", "dtype")
    return {k: line[k] for k in keep if k in line}


def run_prefill(args):
    print(json.dumps(measure_prefill(args, args.steps, args.warmup)), flush=True)


def measure_prefill(args, steps, warmup):
    """Large-batch prefill: T = 4096 tokens through one Gemma-shape layer,
    repeated 30 times (each repetition reads the previous one's output, with
    pre-norm and residual).  One step = 30 layer calls."""
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    shape = synth.GEMMA
    T, R = 4096, (args.layers if args.workload == "prefill" and args.layers else 30)
    layer = make_layers(shape, "prefill", 1, "cuda")[0]
    h = moe.moe_create(shape, [layer], max_tokens=T)
    x = synth.make_tokens(shape, "prefill", T, index=rank).cuda()
    bufs = [torch.empty_like(x), torch.empty_like(x)]
    flags = moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL

    def step():
        src = x
        for r in range(R):
            moe.moe_layer_forward(h, 0, src, bufs[r & 1], flags=flags)
            src = bufs[r & 1]

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    moe.moe_prefill_phase_ms(h)  # clear
    moe.moe_trace_enable(h, True)   # phase events on the launching stream
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    moe.moe_trace_enable(h, False)
    ms = t0.elapsed_time(t1) / steps
    phases, calls = moe.moe_prefill_phase_ms(h)
    per_call = [v / max(calls, 1) for v in phases]
    fl = gemm_flops_per_layer(shape, T)
    gemm_ms = per_call[2] + per_call[3]
    hbm, bf16, src = peaks()
    value = T / (ms / 1e3)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": steps,
        "warmup": warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f16 x f16 -> f32 (tcgen05 kind::f16), 4-bit weights",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 tokens)",
        "config": {"workload": "large prefill: 4096 tokens, one Gemma-shape MoE layer repeated %d "
                               "times, router-driven uniform routing" % R,
                   "tokens_per_step": T, "layer_calls_per_step": R,
                   "l2": "inputs larger than L2: 439 MB of weights per layer call"},
        "phase_ms_per_layer": dict(zip(["router", "bucket", "gemm_gate_up", "gemm_down", "combine"],
                                       per_call)),
        "roofline": {"bound": "tensor", "kernel": "gemm_tc_kernel (gate/up + down launches)",
                     "achieved": fl / (gemm_ms / 1e3) / 1e12, "peak": bf16,
                     "peak_source": src + " bf16 dense (fp16 dense has the same nominal rate)",
                     "unit": "TFLOP/s", "frac": fl / (gemm_ms / 1e3) / 1e12 / bf16,
                     "flops_per_layer": fl, "avg_gemm_ms_per_layer": gemm_ms, "traffic": None},
        "layer_tflops": (fl + 2 * T * shape.n_experts * shape.d_model) / (ms / R / 1e3) / 1e12,
        "whole_layer": {"ms": ms / R, "flops": fl + 2 * T * shape.n_experts * shape.d_model,
                        "tflops": (fl + 2 * T * shape.n_experts * shape.d_model) / (ms / R / 1e3) / 1e12,
                        "frac": (fl + 2 * T * shape.n_experts * shape.d_model) / (ms / R / 1e3)
                                / 1e12 / bf16,
                        "peak": bf16, "peak_source": src + " bf16 dense, burst"},
        "clocks": clk,
    }
    moe.moe_destroy(h)
    del layer
    torch.cuda.empty_cache()
    return line


def run_chunked(args):
    print(json.dumps(measure_chunked(args, args.steps, args.warmup)), flush=True)


def measure_chunked(args, steps, warmup):
    """Chunked prefill: 1024 tokens in 8 chunks of 128 through the 30-layer
    stack, router biased so expert popularity follows Zipf(1.1).  One step =
    8 chunks x 30 layers."""
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    shape = synth.GEMMA
    L = (args.layers if args.workload == "chunked_prefill" and args.layers else shape.n_layers)
    out = []
    for l in range(L):
        Lw = synth.make_layer(shape, "chunked_prefill", l, device="cuda", logit_bias=True)
        out.append(synth.layer_to(Lw, "cpu"))
        del Lw
    torch.cuda.empty_cache()
    h = moe.moe_create(shape, out, max_tokens=128)
    x = synth.make_tokens(shape, "chunked_prefill", 1024, index=rank).cuda()
    y = torch.empty_like(x)

    def step():
        for c in range(8):
            moe.moe_forward_stack(h, x[c * 128:(c + 1) * 128], y[c * 128:(c + 1) * 128], L)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # touched expert bytes: distinct experts per (chunk, layer) from the ids
    touched = 0
    for c in range(8):
        moe.moe_forward_stack(h, x[c * 128:(c + 1) * 128], y[c * 128:(c + 1) * 128], L)
        ids, _ = moe.moe_stack_ids(h, L, 128)
        for l in range(L):
            touched += len(np.unique(ids[l])) * shape.expert_bytes()
    touched += 8 * L * (shape.shared_bytes() + shape.router_bytes())
    # phase breakdown of one step (CUDA events between the kernels of each call)
    moe.moe_prefill_phase_ms(h)
    moe.moe_trace_enable(h, True)
    step()
    torch.cuda.synchronize()
    moe.moe_trace_enable(h, False)
    phases, calls = moe.moe_prefill_phase_ms(h)
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / steps
    hbm, bf16, src = peaks()
    gbs = touched / (ms / 1e3) / 1e9
    line = {
        "metric": METRIC, "value": 1024 / (ms / 1e3), "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 x f16 -> f32 (tcgen05 kind::f16), 4-bit weights",
        "data": "synthetic (seeded; Zipf(1.1) router logit bias)",
        "config": {"workload": "chunked prefill: 1024 tokens in 8 chunks of 128 through %d "
                               "layers, Zipf(1.1)-biased routing" % L,
                   "tokens_per_step": 1024},
        "touched_weight_bytes_per_step": touched,
        "phase_ms_per_chunk_layer": dict(zip(["router", "bucket", "gemm_gate_up", "gemm_down",
                                              "combine"], [v / max(calls, 1) for v in phases])),
        "roofline": {"bound": "hbm", "kernel": "whole chunk step (touched weight bytes)",
                     "achieved": gbs, "peak": hbm, "peak_source": src, "unit": "GB/s",
                     "frac": gbs / hbm, "traffic": None},
        "clocks": clk,
    }
    moe.moe_destroy(h)
    del out
    torch.cuda.empty_cache()
    return line


def h2d_link_gbs(device_index: int) -> float:
    """Pinned host -> device copy bandwidth: 1 GiB cudaMemcpyAsync, best of 10."""
    import torch
    n = 1 << 30
    src = torch.empty(n, dtype=torch.uint8, pin_memory=True)
    dst = torch.empty(n, dtype=torch.uint8, device="cuda")
    best = float("inf")
    for _ in range(10):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        dst.copy_(src, non_blocking=True)
        b.record()
        torch.cuda.synchronize()
        best = min(best, a.elapsed_time(b))
    del src, dst
    torch.cuda.empty_cache()
    return n / (best / 1e3) / 1e9


def run_batched(args):
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    L = args.layers or synth.GEMMA.n_layers
    layers = make_layers(synth.GEMMA, "decode", L, "cuda")
    h = moe.moe_create(synth.GEMMA, layers, max_tokens=args.batch)
    del layers
    print(json.dumps(measure_batched(args, h, L, args.batch, args.steps, args.warmup)), flush=True)


def measure_batched(args, h, L, B, steps, warmup):
    """Batched decode: a batch of B tokens (default 32) through the L-layer
    decode stack per step, on the same weights as the decode workload.  From
    5 tokens on, each layer takes the multi-token path (router GEMM,
    bucketing, grouped tensor-core GEMMs, combine), so each chosen expert's
    weights are read once for all the batch's rows routed to it; fewer tokens
    run as one single-token decode launch each (moe_forward_stack decides)."""
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    rank, world, local = dist_env()
    shape = synth.GEMMA
    x = synth.make_tokens(shape, "decode", B, index=3000 + rank).cuda()
    y = torch.empty_like(x)

    def step():
        moe.moe_forward_stack(h, x, y, L)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    # touched expert bytes: distinct experts per layer from the ids
    ids, _ = moe.moe_stack_ids(h, L, B)
    touched = sum(len(np.unique(ids[l])) * shape.expert_bytes() for l in range(L))
    touched += L * (shape.shared_bytes() + shape.router_bytes())
    moe.moe_prefill_phase_ms(h)
    moe.moe_trace_enable(h, True)
    step()
    torch.cuda.synchronize()
    moe.moe_trace_enable(h, False)
    phases, calls = moe.moe_prefill_phase_ms(h)
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    torch.cuda.synchronize()
    t0.record(stream)
    for _ in range(steps):
        step()
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / steps
    value = B / (ms / 1e3)
    hbm, bf16, src = peaks()
    gbs = touched / (ms / 1e3) / 1e9
    multi = B >= 5  # moe_forward_stack's split between the two paths
    per_layer = 8 if B * shape.top_k <= 2048 else 10
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1,
        "steps": steps, "warmup": warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 x f16 -> f32 (tcgen05 kind::f16), 4-bit weights",
        "data": "synthetic (seeded N(0,0.02) weights, N(0,1) bf16 tokens, router-driven ids)",
        "config": {"workload": "batched decode: %d tokens per step through %d layers "
                               "(the decode stack's weights), router-driven routing" % (B, L),
                   "tokens_per_step": B,
                   "l2": "inputs larger than L2: %d MB of touched weights per layer"
                         % round(touched / L / 1e6)},
        "touched_weight_bytes_per_step": touched,
        "path": "multi-token, layer by layer" if multi else "one decode launch per token",
        "phase_ms_per_layer": dict(zip(["router", "bucket", "gemm_gate_up", "gemm_down",
                                        "combine"], [v / max(calls, 1) for v in phases]))
                              if multi else None,
        "roofline": {"bound": "hbm", "kernel": "whole step (touched weight bytes)",
                     "achieved": gbs, "peak": hbm, "peak_source": src, "unit": "GB/s",
                     "frac": gbs / hbm, "traffic": None},
        "gpu_launches": (per_layer * L if multi else B) * steps,
        "clocks": clk,
    }
    return line


def run_streaming(args):
    L = args.layers or 30
    print(json.dumps(measure_streaming(args, args.steps, args.warmup, L, args.store)), flush=True)


def measure_streaming(args, steps, warmup, L, store_dir=None, cpu_baseline=True):
    """Streaming decode with the expert-slot cache: the L x 128 routed experts
    live in a pinned host pool (or, with store_dir, in an expert store file
    written there and read with bounded parallel pread on each miss), each
    layer has 16 HBM slots under LFU, and the top-8 ids of each (step, layer)
    come from a Zipf(1.1) trace that keeps 4 of the previous step's ids.  One
    step = one token through the L layers; the misses are fetched while the
    shared expert runs."""
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    shape = synth.GEMMA
    n_slots = 16
    link = h2d_link_gbs(local)
    layers = make_layers(shape, "streaming_decode", L, "cuda")
    store_path = None
    t_write = 0.0
    if store_dir:
        os.makedirs(store_dir, exist_ok=True)
        store_path = os.path.join(store_dir, "experts_%d_%d.moestore" % (os.getpid(), L))
        t0 = time.perf_counter()
        moe.moe_store_write(shape, layers, store_path)
        t_write = time.perf_counter() - t0
    h = moe.moe_create(shape, layers, n_slots=n_slots, max_tokens=1, expert_store=store_path,
                       io_threads=args.io_threads)
    del layers
    info = moe.moe_get_info(h)
    blob = info["expert_blob_bytes"]
    W, K = warmup, steps
    n = W + 2 * K
    traces = [synth.streaming_trace(shape.n_experts, shape.top_k, n, 1.1, 4,
                                    seed=synth.seed_of(3, l, 9)) for l in range(L)]
    xs = synth.make_tokens(shape, "streaming_decode", n, index=rank)
    xs_dev = xs.cuda()
    bufs = [torch.empty_like(xs_dev[0:1]) for _ in range(2)]
    flags = moe.MOE_FWD_PRENORM | moe.MOE_FWD_RESIDUAL

    def step(i, x):
        hits = misses = 0
        src = x
        for l in range(L):
            st = moe.moe_layer_forward(h, l, src, bufs[l & 1], flags=flags,
                                       forced_ids=traces[l][i:i + 1])
            hits += st["hits"]
            misses += st["misses"]
            src = bufs[l & 1]
        return src, hits, misses

    for i in range(W):
        step(i, xs_dev[i:i + 1])
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    hits = misses = 0
    t0.record(stream)
    for i in range(W, W + K):
        _, a, b = step(i, xs_dev[i:i + 1])
        hits += a
        misses += b
    t1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = t0.elapsed_time(t1) / K
    # compute alone: the same launches with every id resident (the step-0
    # ids of each layer repeated: all hits after the first step)
    def step_hits(x):
        src = x
        for l in range(L):
            moe.moe_layer_forward(h, l, src, bufs[l & 1], flags=flags, forced_ids=traces[l][0:1])
            src = bufs[l & 1]

    moe.moe_cache_reset(h)
    step_hits(xs_dev[0:1])
    torch.cuda.synchronize()
    c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    c0.record(stream)
    for i in range(K):
        step_hits(xs_dev[i:i + 1])
    c1.record(stream)
    torch.cuda.synchronize()
    ms_compute = c0.elapsed_time(c1) / K
    moe.moe_cache_reset(h)
    # end to end: x from pinned host memory, y back to the host, every step
    xs_pin = xs.pin_memory()
    y_host = torch.empty((1, shape.d_model), dtype=torch.bfloat16, pin_memory=True)
    torch.cuda.synchronize()
    te0 = time.perf_counter()
    for i in range(W + K, W + 2 * K):
        xd = xs_pin[i:i + 1].to("cuda", non_blocking=True)
        out, _, _ = step(i, xd)
        y_host.copy_(out, non_blocking=True)
    torch.cuda.synchronize()
    te = (time.perf_counter() - te0) / K
    h2d = misses * blob / K  # bytes per step
    value = 1e3 / ms
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": 1, "steps": K,
        "warmup": W, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u4 x s16 -> s32 (dp2a) per 32-column chunk, f32 scale and sum",
        "data": "synthetic (seeded; forced ids from a Zipf(1.1) trace, 4 of 8 kept per step)",
        "config": {"workload": "streaming decode: %d layers, 16 HBM slots per layer under LFU, "
                               "routed experts in a %.2f GB %s, %d decode steps"
                               % (L, L * shape.n_experts * blob / 1e9,
                                  "expert store file read with pread" if store_path
                                  else "pinned host pool", K),
                   "layers": L, "n_slots": n_slots, "tokens_per_step": 1,
                   "l2": "inputs larger than L2: 1.12 GB of weights per token"},
        "hit_rate": hits / max(hits + misses, 1),
        "misses_per_layer_step": misses / (K * L),
        "h2d_bytes_per_step_weights": h2d,
        "h2d_gbs": h2d / (ms / 1e3) / 1e9,
        "h2d_link_gbs": link,
        "roofline": {"bound": "h2d", "kernel": "expert miss copies (side stream)",
                     "achieved": h2d / (ms / 1e3) / 1e9, "peak": link,
                     "peak_source": "measured here: pinned 1 GiB cudaMemcpyAsync, best of 10",
                     "unit": "GB/s", "frac": h2d / (ms / 1e3) / 1e9 / link, "traffic": None},
        # copies alone (the step's miss bytes at the measured link rate), compute
        # alone (all hits) and the step: 1 = the fetches are fully hidden under
        # the compute (or the compute under them), 0 = they run one after the other
        "overlap": {"fetch_ms": (h2d / (link * 1e9) * 1e3 if not store_path else None),
                    "compute_ms": ms_compute, "step_ms": ms,
                    "efficiency": (max(0.0, min(1.0, (h2d / (link * 1e9) * 1e3 + ms_compute - ms)
                                                / min(h2d / (link * 1e9) * 1e3, ms_compute)))
                                   if not store_path and h2d > 0 else None)},
        "e2e": {"value": 1.0 / te, "unit": "tokens/s", "h2d_bytes_per_step": 2 * shape.d_model,
                "d2h_bytes_per_step": 2 * shape.d_model, "api": "moe_layer_forward x 30"},
        "gpu_launches": 2 * L * K,
        "clocks": clk,
    }
    if store_path:
        line["store"] = {"path_dir": store_dir, "direct_io": bool(info["store_direct_io"]),
                         "io_threads": info["io_threads"], "write_s": t_write,
                         "read_gbs": h2d / (ms / 1e3) / 1e9}
    moe.moe_destroy(h)
    if store_path:
        os.unlink(store_path)
    if cpu_baseline and not args.no_cpu_baseline:
        import oracle
        layers_cpu = make_layers(shape, "streaming_decode", min(L, 4), "cuda")
        t_c = time.perf_counter()
        done = 0
        x = xs[0:1]
        lfus = [oracle.LFUCache(n_slots, shape.n_experts) for _ in range(len(layers_cpu))]
        while time.perf_counter() - t_c < args.cpu_budget and done < len(layers_cpu):
            lfus[done].step(traces[done][0])
            ref = oracle.moe_layer(oracle.LayerView(shape, layers_cpu[done]), x,
                                   traces[done][0:1], prenorm=True)
            x = (x.float() + torch.tensor(ref["y"], dtype=torch.float32)).to(torch.bfloat16)
            done += 1
        dt = time.perf_counter() - t_c
        line["cpu_baseline"] = {"value": 1.0 / (dt / done * L), "unit": "tokens/s",
                                "cores": os.cpu_count(), "kind": "oracle",
                                "sample": "one token through %d layers with the LFU replay "
                                          "(%.1f s), scaled to %d layers" % (done, dt, L)}
    torch.cuda.empty_cache()
    return line


TRACE_NAMES = ["start", "input_reduced", "routed", "bs_ready", "bs_done", "br_first_ready",
               "br_last_ready", "br_done", "h_complete", "h_converted", "c_first_ready", "c_done",
               "next_barrier"]


def run_trace(args):
    """Per-phase device trace of one decode launch: the median over CTAs of
    each phase's duration (us), per layer, from the kernel's %globaltimer
    stamps (moe_trace_enable / moe_trace_read)."""
    import torch
    import synth
    import expert_ffn_streaming_bit_b300 as moe
    torch.cuda.set_device(0)
    shape = synth.GEMMA
    L = args.layers or 4
    layers = make_layers(shape, "decode", L, "cuda")
    h = moe.moe_create(shape, layers, max_tokens=1)
    x = synth.make_tokens(shape, "decode", 1, index=5).cuda()
    y = torch.empty_like(x)
    for _ in range(5):
        moe.moe_forward_stack(h, x, y, L)
    torch.cuda.synchronize()
    moe.moe_trace_enable(h, True)
    moe.moe_forward_stack(h, x, y, L)
    torch.cuda.synchronize()
    tr = moe.moe_trace_read(h, L).astype(np.float64)
    moe.moe_trace_enable(h, False)
    for l in range(L):
        d = np.diff(tr[:, l, :], axis=1) / 1000.0
        phases = {TRACE_NAMES[e + 1]: round(float(np.median(d[:, e])), 3) for e in range(d.shape[1])
                  if np.all(np.isfinite(d[:, e])) and np.median(d[:, e]) >= 0}
        print(json.dumps({"layer": l, "phase_us_median_over_ctas": phases}), flush=True)


def run_reference(args):
    """The oracle as it stands on the host cores, on the decode workload: one
    step = one token through all the layers (pre-norm and residual between
    layers, as the GPU arm's stack)."""
    rank, world, local = dist_env()
    if rank != 0:
        return
    import torch
    import synth
    import oracle
    shape = synth.GEMMA
    L = args.layers or shape.n_layers
    device = "cuda" if torch.cuda.is_available() else "cpu"
    layers = make_layers(shape, "decode", L, device)
    xs = synth.make_tokens(shape, "decode", args.warmup + args.steps, index=4000)
    cores = oracle.set_threads(os.cpu_count() or 1)

    def token(i):
        dt, n = oracle_sample(shape, layers, xs[i:i + 1], float("inf"))
        assert n == L
        return dt

    for i in range(args.warmup):
        token(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        token(args.warmup + i)
    dt = time.perf_counter() - t0
    per_token = dt / args.steps
    value = 1.0 / per_token
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": per_token * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,0.02) weights quantised to affine 4-bit g64; N(0,1) bf16 tokens)",
        "config": decode_config(L, 1),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "each step: one token through all %d layers (fp64 C oracle, "
                                   "OpenMP over rows)" % L},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None,
                    help="timed steps (default: decode 5000, prefill 3, chunked_prefill 2, "
                         "streaming_decode 256, batched_decode 200)")
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling)")
    ap.add_argument("--cpu-budget", type=float, default=10.0,
                    help="seconds of oracle work per CPU-baseline sample (all cores, 1 core)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sub-records", action="store_true",
                    help="decode line only, without the prefill and chunked-prefill sub-records")
    ap.add_argument("--trace", action="store_true",
                    help="print the decode kernel's per-phase device trace instead of timing")
    ap.add_argument("--workload", default="decode",
                    choices=["decode", "prefill", "chunked_prefill", "streaming_decode",
                             "batched_decode", "layer_step"],
                    help="decode (default, the headline line), a prefill workload, "
                         "streaming decode with the expert-slot cache, or batched decode")
    ap.add_argument("--batch", type=int, default=32, help="tokens per step of batched_decode")
    ap.add_argument("--context", type=int, default=4096,
                    help="layer_step: earlier tokens in the KV caches")
    ap.add_argument("--store", default=None,
                    help="streaming_decode: directory for an expert store file to stream from "
                         "(default: the pinned host pool)")
    ap.add_argument("--io-threads", type=int, default=8,
                    help="expert store: concurrent pread calls per miss batch")
    args = ap.parse_args()
    if args.steps is None:
        args.steps = {"decode": 5000, "prefill": 3, "chunked_prefill": 2,
                      "streaming_decode": 256, "batched_decode": 200,
                      "layer_step": 100}[args.workload]
        if args.impl == "reference":
            args.steps = 20
    if args.warmup < 3:
        args.warmup = 3
    if args.trace:
        run_trace(args)
        return
    if args.impl == "reference":
        if args.steps > 20:
            args.steps = 20   # each reference step is one token through the whole stack
        run_reference(args)
    elif args.workload == "prefill":
        run_prefill(args)
    elif args.workload == "chunked_prefill":
        run_chunked(args)
    elif args.workload == "streaming_decode":
        run_streaming(args)
    elif args.workload == "batched_decode":
        run_batched(args)
    elif args.workload == "layer_step":
        run_layer_step(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
