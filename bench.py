"""Decode throughput of the batch-invariant Qwen3-8B-shaped forward step.

One step = one decode iteration for every request of the batch: embedding
gather, 36 decoder layers (RMSNorm, QKV GEMM, RoPE + KV append, split-KV
attention, O GEMM, residual RMSNorm, gate/up GEMM with SwiGLU in its epilogue,
down GEMM), final RMSNorm, LM head GEMM (fp32 logits), seeded sampler,
position/history update.
Weights are random ~N(0, 0.02) bf16 (gains 1), the prompt KV cache ~N(0, 1)
bf16 for prompt lengths drawn U{16..4096}; the step is replayed from a CUDA
graph.  Weights (15 GB per step) exceed L2, so every step streams them from
HBM.

Prints one JSON line (rank 0).  --impl reference times the CPU oracle instead.
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

METRIC = "decode tokens/s (8B-shaped, batch 1-256) and % of HBM / tensor-core roofline"
UNIT = "tokens/s"

# DRAM bytes (read + write) per launch of each GEMM projection at batch 16,
# from one `ncu --set full` capture (profiles/gemm_kernel_qwen3_8b_decode_b16.md).
# Reported only while the GEMM's sources still hash to `src`.
NCU_GEMM_TRAFFIC = {
    "src": "6bb866ca61d7c8c9",
    "batch": 16,
    "bytes": {"gemm_qkv": 50.590e6, "gemm_o": 33.899e6, "gemm_gate_up": 204.416e6,
              "gemm_down": 104.013e6, "gemm_lm_head": 1251.766e6},
}


def _peaks():
    """(HBM GB/s, bf16 TFLOP/s burst, bf16 TFLOP/s sustained, kind): the
    measured copy bandwidth and cuBLAS bf16 rates of the GB300s, else
    the fallback figures."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return (d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0),
                d.get("bf16_tflops_sustained", 1700.0), "measured")
    return 6800.0, 1900.0, 1700.0, "fallback"


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------- replicas (one per GPU)
def max_over_ranks(x: float, device) -> float:
    """The slowest replica's time (no-op with one process)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return x
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def replica_tokens_per_s(batch: int, world: int, ms: float) -> float:
    """Whole-job throughput: every replica decodes `batch` tokens per step."""
    return batch * world / (ms / 1e3)


def replica_lengths(batch: int, rank: int) -> list:
    """Prompt lengths U{16..4096} of one replica's requests (seeded per rank)."""
    from invariant_deterministic_gb300 import synth
    return synth.uniform_int(batch, 16, 4096, synth.SEED_LEN + 100 * rank).tolist()


class Clocks:
    """nvidia-smi sampled while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.proc = None
        self.index = index

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        load = [s for s in sm if s > 0.5 * (max(sm) if sm else 1)]
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------- workload
def build_workload(max_batch, steps_total, n_layers, rank, device, max_chunk=0):
    import torch
    from invariant_deterministic_gb300 import kinv, model as M, synth
    shape = M.ModelShape(**{**M.QWEN3_8B.__dict__, "n_layers": n_layers})
    w = M.random_weights(shape, seed=synth.SEED_WEIGHTS, device=device)
    lens = replica_lengths(max_batch, rank)
    lmax = 4096 + steps_total + 8
    dec = M.Decoder(shape, w, max_batch=max_batch, max_len=lmax, max_chunk=max_chunk, device=device)
    g = synth.gen(synth.SEED_ACT + 100 * rank, device)
    for li in range(n_layers):
        dec.kv[li].normal_(generator=g)   # prompt KV ~N(0, 1)
    base = dict(temperature=0.8, top_k=50, top_p=0.95, min_p=0.05, repeat_penalty=1.1,
                repeat_last_n=64)
    dec.set_sampling([kinv.SamplingParams(**base, seed=synth.SEED_REQ_BASE + 10000 * rank + b)
                      for b in range(max_batch)])
    hist = torch.randint(0, shape.vocab, (max_batch, 64), generator=synth.gen(synth.SEED_LEN + 7 + rank))
    dec.set_history(hist.tolist())
    dec.set_positions(lens)
    dec.tokens[:max_batch].copy_(hist[:, -1].to(torch.int32))
    torch.cuda.synchronize()
    return shape, w, dec, lens


def step_bytes(shape, bsz, lens_now):
    """Algorithmic HBM bytes of one decode step: every weight once, the KV
    cache each request reads (its cached positions plus the new one) and
    writes (the new position), activations and logits."""
    d, hq, hk, dh, f, v = shape.d_model, shape.n_q, shape.n_kv, shape.head_dim, shape.ffn, shape.vocab
    per_layer_w = (shape.qkv_dim * d + d * hq * dh + 2 * f * d + d * f) * 2 + 2 * d * 2
    weights = shape.n_layers * per_layer_w + v * d * 2 + bsz * d * 2 + d * 2
    kv_pos = hk * dh * 2 * 2 * shape.n_layers
    kv = sum((l + 1) * kv_pos for l in lens_now) + bsz * kv_pos
    logits = bsz * v * 4 * 2
    return weights + kv + logits


def workload_name(layers, bsz):
    return (f"Qwen3-8B-shaped decode step ({layers} layers, d 4096, 32/8 heads of 128, FFN 12288, "
            f"vocab 151936), batch {bsz}, prompt lengths U{{16..4096}}, sampler T 0.8 top_k 50 "
            "top_p 0.95 min_p 0.05 repeat penalty 1.1 over 64")


def gemm_bytes(m, n, k, out_bytes=2):
    return (m * k + n * k) * 2 + m * n * out_bytes


def run_prefill(dec, shape, chunk, prompt_len, stream, tc_peak):
    """Chunked prefill of one prompt of `prompt_len` synthetic tokens through
    every layer (sequence slot 0), chunks of `chunk` rows.  Returns tokens/s
    and the tensor-core roofline of the GEMMs (fp32-accumulated bf16 flops
    over the GEMM kernels' own time, from an instrumented pass) and of the
    whole pass (GEMM + attention flops over the wall time)."""
    import torch
    from invariant_deterministic_gb300 import kinv, synth
    ids = torch.randint(0, shape.vocab, (prompt_len,), generator=synth.gen(synth.SEED_LEN + 99))
    ids = ids.to(torch.int32).to(dec.dev)

    def one_pass():
        for p0 in range(0, prompt_len, chunk):
            n = min(chunk, prompt_len - p0)
            kinv.embed(dec.w["embed"], ids[p0: p0 + n], out=dec.x[:n])
            dec.prefill_chunk(0, p0, n)
            dec.close_residual(n)

    with torch.cuda.stream(stream):
        one_pass()                      # warm-up
        stream.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        one_pass()
        t1.record(stream)
        stream.synchronize()
        ms = t0.elapsed_time(t1)
        timer = {}
        dec.timer = timer
        one_pass()
        dec.timer = None
        stream.synchronize()
    d, f, hq, hk, dh = shape.d_model, shape.ffn, shape.n_q, shape.n_kv, shape.head_dim
    lin_per_tok = 2 * (shape.qkv_dim * d + d * hq * dh + 2 * f * d + d * f) * shape.n_layers
    attn_flops = 4 * hq * dh * sum(p + 1 for p in range(prompt_len)) * shape.n_layers
    gemm_ms = sum(a.elapsed_time(b) for k, v in timer.items() if k.startswith("gemm") for a, b in v)
    gemm_tflops = lin_per_tok * prompt_len / (gemm_ms / 1e3) / 1e12
    all_tflops = (lin_per_tok * prompt_len + attn_flops) / (ms / 1e3) / 1e12
    return {"chunk": chunk, "prompt_len": prompt_len, "ms": round(ms, 3),
            "tokens_per_s": round(prompt_len / (ms / 1e3), 1),
            "gemm": {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": tc_peak,
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / tc_peak, 4),
                     "ms": round(gemm_ms, 3)},
            "whole_pass": {"achieved": round(all_tflops, 1), "unit": "TFLOP/s",
                           "frac": round(all_tflops / tc_peak, 4)},
            # per stage, from the instrumented (serialised) pass
            "stage_ms": {k: round(sum(a.elapsed_time(b) for a, b in v), 3) for k, v in sorted(timer.items())}}


def run_kinv(args):
    import torch
    import torch.distributed as dist
    from invariant_deterministic_gb300 import build, kinv, model as M
    build.build()
    ws, rank, local = _dist()
    if ws > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    sweep = sorted(set([args.batch] + [int(x) for x in args.sweep.split(",") if x]))
    bmax = max(sweep)
    # decode steps a row may take: per sweep batch two eager warm-ups, the
    # graph's warm-up and timed replays; then the instrumented pass and the
    # end-to-end warm-up and timed steps
    per_b = args.warmup + args.steps + 3
    steps_total = per_b * len(sweep) + args.prof_steps + args.warmup + args.steps + 8
    shape, w, dec, lens0 = build_workload(bmax, steps_total, args.layers, rank, dev,
                                          max_chunk=max(args.prefill_chunks) if args.prefill else 0)
    hbm_peak, tc_peak, tc_sustained, peak_kind = _peaks()
    # per layer: QKV (+ RoPE/append for M.FUSED_ROPE_MIN_ROWS .. MAX rows, else
    # a separate RoPE/append kernel), attention split + merge, O, gate/up, down;
    # per step: embed, row sums of squares, LM head, sampler, position update
    fused_rope = M.FUSED_ROPE_MIN_ROWS <= args.batch <= M.FUSED_ROPE_MAX_ROWS
    launches_per_step = (6 if fused_rope else 7) * shape.n_layers + 5

    def barrier():
        if ws > 1:
            dist.barrier()

    results = {}
    clocks = None
    stream = torch.cuda.Stream(device=dev)
    for bsz in sweep:
        # warm-up, then capture one step into a graph
        with torch.cuda.stream(stream):
            for _ in range(2):
                dec.decode_step(bsz)
            stream.synchronize()
            assert kinv.last_device_status(stream) == 0
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=stream):
                dec.decode_step(bsz)
            for _ in range(args.warmup):
                graph.replay()
            stream.synchronize()
            lens_now = dec.pos[:bsz].cpu().tolist()
            clk = Clocks(local) if bsz == args.batch else None
            if clk:
                clk.start()
                time.sleep(0.3)
            barrier()
            torch.cuda.synchronize()
            t0 = torch.cuda.Event(enable_timing=True)
            t1 = torch.cuda.Event(enable_timing=True)
            t0.record(stream)
            for _ in range(args.steps):
                graph.replay()
            t1.record(stream)
            torch.cuda.synchronize()
            barrier()
            ms = max_over_ranks(t0.elapsed_time(t1) / args.steps, dev)
            if clk:
                clocks = clk.stop()
            status = kinv.last_device_status(stream)
            if status != 0:
                raise RuntimeError(f"device status {status} after timed steps")
            nbytes = step_bytes(shape, bsz, [l + args.steps // 2 for l in lens_now])
            results[bsz] = dict(batch=bsz, ms_per_step=ms, tokens_per_s=replica_tokens_per_s(bsz, ws, ms),
                                step_gbs=nbytes / (ms / 1e3) / 1e9,
                                step_hbm_frac=nbytes / (ms / 1e3) / 1e9 / hbm_peak,
                                mean_kv_len=sum(lens_now) / len(lens_now), graph=graph)

    # ---- instrumented pass at the headline batch: per-kernel CUDA events
    # The host enqueues each instrumented step while the stream is held by a
    # device-side sleep, so the kernels then run back to back and each event
    # pair brackets its kernel, not a host launch gap.
    bsz = args.batch
    timer = {}
    with torch.cuda.stream(stream):
        for _ in range(args.prof_steps):
            stream.synchronize()
            torch.cuda._sleep(int(200e6))
            dec.timer = timer
            dec.decode_step(bsz)
            dec.timer = None
        stream.synchronize()
    kernel_ms = {k: sum(a.elapsed_time(b) for a, b in v) / len(v) for k, v in timer.items()}
    kernel_n = {k: len(v) // args.prof_steps for k, v in timer.items()}
    total = {k: kernel_ms[k] * kernel_n[k] for k in kernel_ms}
    d, f = shape.d_model, shape.ffn
    gemm_shapes = {"gemm_qkv": (shape.qkv_dim, d), "gemm_o": (d, shape.n_q * shape.head_dim),
                   "gemm_gate_up": (2 * f, d), "gemm_down": (d, f)}
    gemm_b = {k: gemm_bytes(bsz, n, kk) for k, (n, kk) in gemm_shapes.items()}
    ss_b = bsz * (d // 128) * 4  # per-row partial sums of squares (folded RMSNorm)
    # the gate/up GEMM writes silu(g) * u: F columns, not 2F
    gemm_b["gemm_gate_up"] = (bsz * d + 2 * f * d) * 2 + bsz * f * 2 + ss_b
    gemm_b["gemm_qkv"] += ss_b
    # O and down add into the residual stream: read and write it, write the sums
    for k in ("gemm_o", "gemm_down"):
        gemm_b[k] += bsz * d * 2 + ss_b
    gemm_b["gemm_lm_head"] = gemm_bytes(bsz, shape.vocab, d, 4) + ss_b
    lens_now = dec.pos[:bsz].cpu().tolist()
    attn_b = sum(l * shape.n_kv * shape.head_dim * 4 for l in lens_now) + 2 * bsz * shape.n_q * shape.head_dim * 2
    # the GEMM kernel is one kernel (gemm_kernel) across the five projections
    gemm_time = sum(total[k] for k in gemm_b if k in total)
    gemm_bytes_step = sum(gemm_b[k] * kernel_n.get(k, 0) for k in gemm_b)
    attn_time = total.get("attn_decode", 0.0)
    if gemm_time >= attn_time:
        dom = "gemm_kernel (tcgen05, all projections of the step)"
        achieved = gemm_bytes_step / (gemm_time / 1e3) / 1e9
        per_launch = {k: {"bytes": gemm_b[k], "ms": kernel_ms[k],
                          "gbs": gemm_b[k] / (kernel_ms[k] / 1e3) / 1e9,
                          "frac": gemm_b[k] / (kernel_ms[k] / 1e3) / 1e9 / hbm_peak}
                      for k in gemm_b if k in kernel_ms}
        # per-launch DRAM bytes from the ncu capture, averaged like `achieved`
        # (over the step's GEMM launches), while the GEMM sources are unchanged
        traffic = None
        n_launch = sum(kernel_n.get(k, 0) for k in gemm_b)
        if build.source_hash(["gemm.cu", "rope.cuh"]) == NCU_GEMM_TRAFFIC["src"] and bsz == NCU_GEMM_TRAFFIC["batch"]:
            tb = NCU_GEMM_TRAFFIC["bytes"]
            traffic = round(sum(tb[k] * kernel_n.get(k, 0) for k in tb) / n_launch)
        alg_per_launch = round(gemm_bytes_step / n_launch)
    else:
        dom = "attn_split_kernel + attn_merge_kernel (split-KV decode attention)"
        achieved = attn_b / (kernel_ms["attn_decode"] / 1e3) / 1e9
        per_launch = {"attn_decode": {"bytes": attn_b, "ms": kernel_ms["attn_decode"]}}
        traffic = None
        alg_per_launch = attn_b
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": hbm_peak,
                "unit": "GB/s", "frac": round(achieved / hbm_peak, 4), "traffic": traffic,
                "algorithmic_bytes_per_launch": alg_per_launch,
                "peak_kind": f"{peak_kind} (copy bandwidth)", "per_launch": per_launch,
                "step_share": {k: round(v / sum(total.values()), 4) for k, v in
                               sorted(total.items(), key=lambda kv: -kv[1])}}

    # ---- end to end through the public API with host buffers: every step
    # copies the input token ids from pinned host memory, runs the step and
    # copies the sampled ids back (the copies are nodes of the step's graph),
    # and the host reads them before it feeds them to the next step
    head = results[bsz]
    tok_host = torch.empty(bsz, dtype=torch.int32, pin_memory=True)
    out_host = torch.empty(bsz, dtype=torch.int32, pin_memory=True)
    tok_host.copy_(dec.tokens[:bsz].cpu())
    with torch.cuda.stream(stream):
        io_graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(io_graph, stream=stream):
            dec.tokens[:bsz].copy_(tok_host, non_blocking=True)
            dec.decode_step(bsz)
            out_host.copy_(dec.tokens[:bsz], non_blocking=True)
        for _ in range(args.warmup):
            io_graph.replay()
            stream.synchronize()
            tok_host.copy_(out_host)
        barrier()
        stream.synchronize()
        t_start = time.perf_counter()
        for _ in range(args.steps):
            io_graph.replay()
            stream.synchronize()
            tok_host.copy_(out_host)
        e2e_s = max_over_ranks(time.perf_counter() - t_start, dev)
        if kinv.last_device_status(stream) != 0:
            raise RuntimeError("device status after the end-to-end steps")
    e2e = {"value": round(bsz * ws * args.steps / e2e_s, 2), "unit": UNIT,
           "h2d_bytes_per_step": bsz * 4, "d2h_bytes_per_step": bsz * 4}

    # ---- chunked prefill (tensor-core bound) after the decode measurements
    # (a pass of this length runs under the power cap: the sustained peak)
    prefill = None
    if args.prefill:
        prefill = [run_prefill(dec, shape, c, args.prefill_len, stream, tc_sustained)
                   for c in args.prefill_chunks]

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = oracle_full_step(min(args.cpu_rows, bsz), w, dec, shape)
    for r in results.values():
        r.pop("graph", None)
    del dec, w, graph
    torch.cuda.synchronize()
    torch.cuda.empty_cache()

    # stand-alone kernel lines: the projection GEMMs over M and decode
    # attention (+ RMSNorm) over the batch, each launch timed cold
    sweeps = None
    if args.sweeps:
        sweeps = {"gemm": run_gemm_sweep(dev, hbm_peak, tc_peak, peak_kind),
                  "attention": run_attention_sweep(dev, hbm_peak, peak_kind)}
    cpu_configs = None
    if rank == 0 and not args.no_cpu and args.sweeps:
        cpu_configs = oracle_configs()
    line = {
        "metric": METRIC, "value": round(head["tokens_per_s"], 2), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(head["ms_per_step"], 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: random-init weights ~N(0,0.02) bf16, prompt KV cache ~N(0,1) bf16",
        "config": {"workload": workload_name(shape.n_layers, bsz),
                   "batch": bsz, "layers": shape.n_layers, "split_len": 256,
                   "mean_kv_len": round(head["mean_kv_len"], 1), "graph": "CUDA graph per step",
                   "l2": "inputs larger than L2 (15 GB of weights streamed per step)",
                   "parallelism": f"replicas x{ws}"},
        "step_roofline": {"bytes": step_bytes(shape, bsz, lens_now), "gbs": round(head["step_gbs"], 1),
                          "frac": round(head["step_hbm_frac"], 4)},
        "roofline": roofline,
        "prefill": prefill,
        "kernels": sweeps,
        "cpu_baseline": cpu,
        "cpu_configs": cpu_configs,
        "e2e": e2e,
        "gpu_launches": launches_per_step * args.steps,
        "clocks": clocks,
        "sweep": [{k: (round(v, 4) if isinstance(v, float) else v) for k, v in r.items()}
                  for r in results.values()],
        "build_id": kinv.build_id(), "device_class": kinv.device_class(),
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if ws > 1:
        dist.destroy_process_group()


# ---------------------------------------------------------------- the oracle
def _oshape(shape):
    from oracle.model import Shape
    return Shape(d_model=shape.d_model, n_q=shape.n_q, n_kv=shape.n_kv, head_dim=shape.head_dim,
                 ffn=shape.ffn, vocab=shape.vocab, n_layers=shape.n_layers, eps=shape.eps,
                 rope_base=shape.rope_base, qk_norm=shape.qk_norm)


def oracle_full_step(rows, w, dec, shape):
    """Times the CPU oracle on a bounded sample of the same workload: the
    first `rows` requests of the batch (their token, prompt caches and
    positions) through every decoder layer, the final norm, the LM head and
    the sampler -- one whole decode step for those requests, measured, not
    scaled.  The weights and caches are copied to the host before each
    layer's timed region.  Returns the cpu_baseline object."""
    import numpy as np
    from invariant_deterministic_gb300 import synth
    from oracle.glue import embed
    from oracle.model import final_logits, layer_step
    from oracle.sampler import SamplingParams as OP, sample as osample

    cores = len(os.sched_getaffinity(0))
    oshape = _oshape(shape)
    pos = dec.pos[:rows].cpu().tolist()
    lmax = max(pos) + 1
    toks = dec.tokens[:rows].cpu().tolist()
    hist = dec.history[:rows].cpu().tolist()
    params = [OP(temperature=0.8, top_k=50, top_p=0.95, min_p=0.05, repeat_penalty=1.1, repeat_last_n=64,
                 seed=synth.SEED_REQ_BASE + b) for b in range(rows)]
    table = synth.bits(w["embed"])
    t_total = 0.0
    t0 = time.perf_counter()
    x = embed(table, toks)
    t_total += time.perf_counter() - t0
    del table
    for li in range(shape.n_layers):
        lw = {k: synth.bits(v) for k, v in w["layers"][li].items()}
        kc = synth.bits(dec.kv[li, 0, :rows, :lmax])
        vc = synth.bits(dec.kv[li, 1, :rows, :lmax])
        t0 = time.perf_counter()
        x = layer_step(x, lw, kc, vc, [(b, pos[b]) for b in range(rows)], oshape)
        t_total += time.perf_counter() - t0
    head = {"lm_head": synth.bits(w["lm_head"]), "final_norm": synth.bits(w["final_norm"])}
    t0 = time.perf_counter()
    logits = final_logits(x, head, oshape)
    osample(logits, hist, [0] * rows, params)
    t_total += time.perf_counter() - t0
    return {"value": round(rows / t_total, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"the batch's first {rows} requests through one whole decode step (embedding, "
                      f"{shape.n_layers} decoder layers, final norm, LM head, sampler), fp64 NumPy oracle; "
                      "measured, not scaled",
            "seconds": round(t_total, 2)}


def oracle_configs():
    """The oracle timed on the kernel-level workloads (CPU, fp64): the small
    decoder layer over batch 1-4 x KV lengths 1-64 (in full), the four
    8B-shaped projection GEMMs at every M of the sweep (in full), and decode
    attention + RMSNorm for 8 sequences with KV lengths U{1..32768} (a
    bounded sample of the 1-128 sweep)."""
    import numpy as np
    import torch
    from invariant_deterministic_gb300 import synth
    from oracle import attention as oattn
    from oracle.gemm import gemm as ogemm
    from oracle.model import Shape, layer_step
    from oracle.rmsnorm import rmsnorm as ormsnorm
    out = []
    # small layer, every (B, L)
    tiny = Shape(d_model=256, n_q=4, n_kv=2, head_dim=64, ffn=512, eps=1e-6, rope_base=1e4)
    lw = {k: synth.bits(v) for k, v in synth.layer_weights(256, 4, 2, 64, 512, 0, False).items()}
    kc0 = synth.bits(synth.normal_bf16((4, 64, 2, 64), 1.0, 1))
    vc0 = synth.bits(synth.normal_bf16((4, 64, 2, 64), 1.0, 2))
    x = synth.bits(synth.normal_bf16((4, 256), 1.0, 3))
    t0 = time.perf_counter()
    n = 0
    for bsz in range(1, 5):
        for L in range(1, 65):
            layer_step(x[:bsz], lw, kc0[:bsz].copy(), vc0[:bsz].copy(), [(b, L - 1) for b in range(bsz)], tiny)
            n += bsz
    dt = time.perf_counter() - t0
    out.append({"workload": "small decoder layer (d 256, 4/2 heads of 64, FFN 512), B 1-4 x L 1-64",
                "rows_per_s": round(n / dt, 1), "seconds": round(dt, 2), "sample": "in full"})
    # projection GEMMs
    flops = 0
    t_g = 0.0
    for name, (nn, kk) in (("qkv", (6144, 4096)), ("o", (4096, 4096)), ("gate_up", (24576, 4096)),
                           ("down", (4096, 12288))):
        wb = synth.bits(synth.normal_bf16((nn, kk), 0.02, 6))
        ab = synth.bits(synth.normal_bf16((256, kk), 1.0, 7))
        for m in (1, 7, 16, 64, 128, 256):
            t0 = time.perf_counter()
            ogemm(ab[:m], wb)
            t_g += time.perf_counter() - t0
            flops += 2 * m * nn * kk
    out.append({"workload": "8B-shaped projection GEMMs (N, K) in {(6144, 4096), (4096, 4096), (24576, 4096), "
                            "(4096, 12288)} x M in {1, 7, 16, 64, 128, 256}",
                "gflop_per_s": round(flops / t_g / 1e9, 2), "seconds": round(t_g, 2), "sample": "in full"})
    # decode attention + RMSNorm, 8 sequences
    lens = synth.uniform_int(8, 1, 32768, synth.SEED_LEN).tolist()
    q = synth.bits(synth.normal_bf16((8, 32, 128), 1.0, 32))
    xs = synth.bits(synth.normal_bf16((8, 4096), 1.0, 33))
    g = synth.bits(torch.ones(4096, dtype=torch.bfloat16))
    t_a, nbytes = 0.0, 0
    for b in range(8):
        k = synth.bits(synth.normal_bf16((1, lens[b], 8, 128), 1.0, 40 + b))
        v = synth.bits(synth.normal_bf16((1, lens[b], 8, 128), 1.0, 50 + b))
        t0 = time.perf_counter()
        oattn.decode(q[b: b + 1], k, v, [lens[b]])
        t_a += time.perf_counter() - t0
        nbytes += lens[b] * 8 * 128 * 2 * 2
    t0 = time.perf_counter()
    ormsnorm(xs, g, 1e-6)
    t_a += time.perf_counter() - t0
    out.append({"workload": "decode attention (32/8 heads of 128, KV lengths U{1..32768}) + RMSNorm (d 4096)",
                "gb_per_s": round(nbytes / t_a / 1e9, 3), "seconds": round(t_a, 2),
                "sample": "8 sequences of the 1-128 sweep (seed 2)"})
    return {"cores": len(os.sched_getaffinity(0)), "kind": "oracle", "configs": out}


# ---------------------------------------------------------- stand-alone kernels
class _Flush:
    """Writes a buffer larger than L2 between timed launches."""
    def __init__(self, dev, nbytes=512 << 20):
        import torch
        self.buf = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def __call__(self):
        self.buf.zero_()


def _time_cold(fn, flush, iters):
    """Median CUDA-event time (ms) of fn() with L2 flushed before each call."""
    import torch
    fn()
    times = []
    for _ in range(iters):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        fn()
        b.record()
        b.synchronize()
        times.append(a.elapsed_time(b))
    return statistics.median(times)


def run_gemm_sweep(dev, hbm_peak, tc_peak, peak_kind, iters=15):
    """The Qwen3-8B-shaped projection GEMMs (kinv_gemm, bf16 out) at
    M in {1, 7, 16, 64, 128, 256}, each launch timed alone with L2 flushed:
    algorithmic bytes 2(MK + NK + MN) and flops 2MNK over the launch time,
    against the measured copy bandwidth and the attainable roofline
    min(bf16 peak, flops/bytes x bandwidth)."""
    import torch
    from invariant_deterministic_gb300 import kinv, synth
    flush = _Flush(dev)
    out = []
    for name, (n, k) in (("qkv", (6144, 4096)), ("o", (4096, 4096)), ("gate_up", (24576, 4096)),
                         ("down", (4096, 12288))):
        w = synth.normal_bf16((n, k), 0.02, 6, dev)
        a = synth.normal_bf16((256, k), 1.0, 7, dev)
        c = torch.empty(256, n, dtype=torch.bfloat16, device=dev)
        for m in (1, 7, 16, 64, 128, 256):
            ms = _time_cold(lambda: kinv.gemm(a[:m], w, out=c[:m]), flush, iters)
            nbytes = 2 * (m * k + n * k + m * n)
            flops = 2 * m * n * k
            gbs = nbytes / (ms / 1e3) / 1e9
            tf = flops / (ms / 1e3) / 1e12
            attainable = min(tc_peak, flops / nbytes * hbm_peak / 1e3)
            out.append({"proj": name, "n": n, "k": k, "m": m, "us": round(ms * 1e3, 2),
                        "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm_peak, 4),
                        "tflops": round(tf, 2), "attainable_tflops": round(attainable, 1),
                        "attainable_frac": round(tf / attainable, 4)})
        del w, a, c
    torch.cuda.empty_cache()
    return {"peak_kind": peak_kind, "hbm_peak_gbs": hbm_peak, "bf16_peak_tflops": tc_peak,
            "timing": "median of per-launch CUDA events, L2 flushed (512 MB write) before each launch",
            "lines": out}


def run_attention_sweep(dev, hbm_peak, peak_kind, iters=7):
    """Decode attention (32 query / 8 kv heads of 128, split 256) with KV
    lengths drawn U{1..32768} for batch 1..128, and the RMSNorm over the
    batch's d = 4096 rows, each timed alone with L2 flushed: algorithmic bytes
    (K and V of every cached position read once, q read, out written) over the
    launch time."""
    import torch
    from invariant_deterministic_gb300 import kinv, synth
    flush = _Flush(dev)
    bmax, lmax = 128, 32768
    g = synth.gen(synth.SEED_ACT, dev)
    k = torch.empty(bmax, lmax, 8, 128, dtype=torch.bfloat16, device=dev).normal_(generator=g)
    v = torch.empty_like(k).normal_(generator=g)
    q = synth.normal_bf16((bmax, 32, 128), 1.0, 32, dev)
    x = synth.normal_bf16((bmax, 4096), 1.0, 33, dev)
    gain = torch.ones(4096, dtype=torch.bfloat16, device=dev)
    y = torch.empty_like(x)
    ws = torch.empty(kinv.attn_decode_workspace(bmax, 32, 128, lmax), dtype=torch.uint8, device=dev)
    out = torch.empty_like(q)
    lines = []
    for bsz in (1, 2, 4, 8, 16, 32, 64, 128):
        lens = synth.uniform_int(bsz, 1, lmax, synth.SEED_LEN).to(dev)
        ms = _time_cold(lambda: kinv.attn_decode(q[:bsz], k[:bsz], v[:bsz], lens, out=out[:bsz], workspace=ws),
                        flush, iters)
        nbytes = int(lens.sum().item()) * 8 * 128 * 2 * 2 + 2 * bsz * 32 * 128 * 2
        ms_n = _time_cold(lambda: kinv.rmsnorm(x[:bsz], gain, 1e-6, out=y[:bsz]), flush, iters)
        nb_n = bsz * 4096 * 2 * 2 + 4096 * 2
        lines.append({"batch": bsz, "kv_positions": int(lens.sum().item()), "attn_us": round(ms * 1e3, 2),
                      "attn_gbs": round(nbytes / (ms / 1e3) / 1e9, 1),
                      "attn_hbm_frac": round(nbytes / (ms / 1e3) / 1e9 / hbm_peak, 4),
                      "rmsnorm_us": round(ms_n * 1e3, 2),
                      "rmsnorm_gbs": round(nb_n / (ms_n / 1e3) / 1e9, 1)})
    assert kinv.last_device_status() == 0
    del k, v, ws
    torch.cuda.empty_cache()
    return {"peak_kind": peak_kind, "hbm_peak_gbs": hbm_peak,
            "timing": "median of per-launch CUDA events, L2 flushed (512 MB write) before each launch",
            "lines": lines}


def run_reference(args):
    """The CPU oracle as the reference arm, on the GPU arm's workload: each
    timed step is one whole decode step of the 36-layer Qwen3-8B-shaped model
    for the batch's first min(batch, 16) requests (embedding, every decoder
    layer, final norm, LM head, sampler), measured, not scaled.  Weights are
    drawn on the host (36 distinct layers, the GPU arm's distributions).  The
    oracle keeps no state to warm, so each untimed warm-up step runs the first
    layer only (it pages the arrays in)."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import numpy as np
    import torch
    from invariant_deterministic_gb300 import synth
    from oracle.glue import embed
    from oracle.model import Shape, final_logits, layer_step
    from oracle.sampler import SamplingParams as OP, sample as osample

    cores = len(os.sched_getaffinity(0))
    n_layers = args.layers
    oshape = Shape(d_model=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288, vocab=151936, n_layers=n_layers,
                   eps=1e-6, rope_base=1e6, qk_norm=True)
    layers = [{k: synth.bits(v) for k, v in synth.layer_weights(4096, 32, 8, 128, 12288, li, True).items()}
              for li in range(n_layers)]
    table = synth.bits(synth.normal_bf16((151936, 4096), 0.02, 997))
    head = {"lm_head": synth.bits(synth.normal_bf16((151936, 4096), 0.02, 998)),
            "final_norm": synth.bits(torch.ones(4096, dtype=torch.bfloat16))}
    bsz = args.batch
    rows = min(bsz, 16)
    lens = replica_lengths(bsz, 0)[:rows]
    lmax = max(lens) + args.steps + 2
    # the requests' prompt caches, per layer ~N(0, 1)
    kcs = [synth.bits(synth.normal_bf16((rows, lmax, 8, 128), 1.0, 100 + li)) for li in range(n_layers)]
    vcs = [synth.bits(synth.normal_bf16((rows, lmax, 8, 128), 1.0, 500 + li)) for li in range(n_layers)]
    hist = [synth.uniform_int(64, 0, 151935, 6000 + r).tolist() for r in range(rows)]
    params = [OP(temperature=0.8, top_k=50, top_p=0.95, min_p=0.05, repeat_penalty=1.1, repeat_last_n=64,
                 seed=synth.SEED_REQ_BASE + r) for r in range(rows)]
    toks = [h[-1] for h in hist]

    def step(i, depth):
        t0 = time.perf_counter()
        x = embed(table, toks)
        pos = [(r, lens[r] + i) for r in range(rows)]
        for li in range(depth):
            x = layer_step(x, layers[li], kcs[li], vcs[li], pos, oshape)
        if depth == n_layers:
            logits = final_logits(x, head, oshape)
            new, _ = osample(logits, hist, [i] * rows, params)
            for r in range(rows):
                hist[r].append(int(new[r]))
                toks[r] = int(new[r])
        return time.perf_counter() - t0

    for _ in range(args.warmup):
        step(0, 1)
    times = [step(i, n_layers) for i in range(args.steps)]
    per_step = sum(times) / len(times)
    value = rows / per_step
    sample = (f"the batch's first {rows} requests through whole {n_layers}-layer decode steps (embedding, "
              "layers, final norm, LM head, sampler), fp64 NumPy oracle; every timed step measured whole, "
              "not scaled; warm-up steps run one layer")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: random-init weights ~N(0,0.02) bf16, prompt KV cache ~N(0,1) bf16",
        "config": {"workload": workload_name(n_layers, bsz), "batch": bsz, "layers": n_layers, "split_len": 256,
                   "parallelism": f"replicas x{ws}"},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def run_case(spec: str, iters: int):
    """One kernel on a small stand-alone case, `iters` launches after one
    warm-up (for profiler captures): gemm:M:N:K (kinv_gemm, bf16 out),
    attn_prefill:T (one sequence's T-row chunk at position 0, 32/8 heads of
    128), attn_decode:B (B sequences, KV lengths U{1..32768}).  Prints the
    mean launch time."""
    import torch
    from invariant_deterministic_gb300 import build, kinv, synth
    build.build()
    kind, *dims = spec.split(":")
    dims = [int(x) for x in dims]
    dev = torch.device("cuda", 0)
    if kind == "gemm":
        m, n, k = dims
        w = synth.normal_bf16((n, k), 0.02, 6, dev)
        a = synth.normal_bf16((m, k), 1.0, 7, dev)
        c = torch.empty(m, n, dtype=torch.bfloat16, device=dev)
        fn = lambda: kinv.gemm(a, w, out=c)
    elif kind == "attn_prefill":
        (t,) = dims
        g = synth.gen(synth.SEED_ACT, dev)
        kc = torch.empty(1, t, 8, 128, dtype=torch.bfloat16, device=dev).normal_(generator=g)
        vc = torch.empty_like(kc).normal_(generator=g)
        q = synth.normal_bf16((t, 32, 128), 1.0, 32, dev)
        i32 = dict(dtype=torch.int32, device=dev)
        st, ln, off = torch.zeros(1, **i32), torch.tensor([t], **i32), torch.zeros(1, **i32)
        out = torch.empty_like(q)
        ws = torch.empty(kinv.attn_prefill_workspace(t, 32, 128, t), dtype=torch.uint8, device=dev)
        fn = lambda: kinv.attn_prefill(q, kc, vc, st, ln, off, t, t, out=out, workspace=ws)
    elif kind == "attn_decode":
        (b,) = dims
        g = synth.gen(synth.SEED_ACT, dev)
        kc = torch.empty(b, 32768, 8, 128, dtype=torch.bfloat16, device=dev).normal_(generator=g)
        vc = torch.empty_like(kc).normal_(generator=g)
        q = synth.normal_bf16((b, 32, 128), 1.0, 32, dev)
        lens = synth.uniform_int(b, 1, 32768, synth.SEED_LEN).to(dev)
        out = torch.empty_like(q)
        ws = torch.empty(kinv.attn_decode_workspace(b, 32, 128, 32768), dtype=torch.uint8, device=dev)
        fn = lambda: kinv.attn_decode(q, kc, vc, lens, out=out, workspace=ws)
    else:
        raise SystemExit(f"unknown case {spec}")
    fn()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(iters):
        fn()
    e1.record()
    torch.cuda.synchronize()
    status = kinv.last_device_status()
    print(json.dumps({"case": spec, "iters": iters, "ms_per_launch": round(e0.elapsed_time(e1) / iters, 4),
                      "device_status": status}), flush=True)
    if status != 0:
        raise SystemExit(1)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kinv", choices=["kinv", "reference"])
    ap.add_argument("--batch", type=int, default=16)
    ap.add_argument("--sweep", default="1,64,256")
    ap.add_argument("--layers", type=int, default=36)
    ap.add_argument("--prof-steps", type=int, default=3)
    ap.add_argument("--cpu-rows", type=int, default=16)
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-sweeps", dest="sweeps", action="store_false")
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--prefill-len", type=int, default=4096)
    ap.add_argument("--prefill-chunks", default="512,4096")
    ap.add_argument("--case", default=None, help="run one kernel case (gemm:M:N:K, attn_prefill:T, attn_decode:B)")
    ap.add_argument("--case-iters", type=int, default=3)
    args = ap.parse_args()
    if args.case:
        run_case(args.case, args.case_iters)
        return
    if args.warmup < 3:
        args.warmup = 3
    args.prefill_chunks = [int(c) for c in str(args.prefill_chunks).split(",") if c]
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kinv(args)


if __name__ == "__main__":
    main()
