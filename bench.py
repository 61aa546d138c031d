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
    "src": "e69e7953411db204",
    "batch": 16,
    "bytes": {"gemm_qkv": 50.593e6, "gemm_o": 33.900e6, "gemm_gate_up": 204.433e6,
              "gemm_down": 104.092e6, "gemm_lm_head": 1250.960e6},
}


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


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
    per_b = args.warmup + args.steps + 3
    shape, w, dec, lens0 = build_workload(bmax, per_b * len(sweep) + 8, args.layers, rank, dev,
                                          max_chunk=max(args.prefill_chunks) if args.prefill else 0)
    hbm_peak, tc_peak, peak_kind = _peaks()
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

    # ---- end to end through the public API with host buffers
    head = results[bsz]
    graph = head["graph"]
    tok_host = torch.empty(bsz, dtype=torch.int32, pin_memory=True)
    out_host = torch.empty(bsz, dtype=torch.int32, pin_memory=True)
    tok_host.copy_(dec.tokens[:bsz].cpu())
    with torch.cuda.stream(stream):
        barrier()
        stream.synchronize()
        t_start = time.perf_counter()
        for _ in range(args.steps):
            dec.tokens[:bsz].copy_(tok_host, non_blocking=True)
            graph.replay()
            out_host.copy_(dec.tokens[:bsz], non_blocking=True)
            stream.synchronize()
            tok_host.copy_(out_host)
        e2e_s = max_over_ranks(time.perf_counter() - t_start, dev)
    e2e = {"value": round(bsz * ws * args.steps / e2e_s, 2), "unit": UNIT,
           "h2d_bytes_per_step": bsz * 4, "d2h_bytes_per_step": bsz * 4}

    # ---- chunked prefill (tensor-core bound) after the decode measurements
    prefill = None
    if args.prefill:
        prefill = [run_prefill(dec, shape, c, args.prefill_len, stream, tc_peak)
                   for c in args.prefill_chunks]

    cpu = None
    if rank == 0 and not args.no_cpu:
        cpu = oracle_sample(min(args.cpu_rows, bsz), w, dec, shape)
    for r in results.values():
        r.pop("graph", None)
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
        "cpu_baseline": cpu,
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
def oracle_sample(rows, w, dec, shape, budget_s=12.0):
    """Times the CPU oracle on a bounded sample of the same workload: `rows`
    requests through as many decoder layers as fit in about `budget_s`
    seconds (at least one), the final norm, the LM head and the sampler;
    the layer time is scaled to the full depth.  Returns the cpu_baseline
    object."""
    import numpy as np
    import torch
    from invariant_deterministic_gb300 import synth
    from oracle.gemm import gemm as ogemm
    from oracle.model import Shape, layer_step
    from oracle.rmsnorm import rmsnorm as ormsnorm
    from oracle.sampler import SamplingParams as OP, sample as osample

    cores = len(os.sched_getaffinity(0))
    os.environ.setdefault("OMP_NUM_THREADS", str(cores))
    oshape = Shape(d_model=shape.d_model, n_q=shape.n_q, n_kv=shape.n_kv, head_dim=shape.head_dim,
                   ffn=shape.ffn, vocab=shape.vocab, n_layers=shape.n_layers, eps=shape.eps,
                   rope_base=shape.rope_base, qk_norm=shape.qk_norm)
    pos = dec.pos[:rows].cpu().tolist()
    lmax = max(pos) + 1
    x = synth.bits(dec.x[:rows])
    head = synth.bits(w["lm_head"])
    fnorm = synth.bits(w["final_norm"])
    layer_s = 0.0
    layers = 0
    while layers < shape.n_layers and (layers == 0 or layer_s < budget_s):
        li = layers
        lw = {k: synth.bits(v) for k, v in w["layers"][li].items()}
        kc = synth.bits(dec.kv[li, 0, :rows, :lmax])
        vc = synth.bits(dec.kv[li, 1, :rows, :lmax])
        t0 = time.perf_counter()
        x = layer_step(x, lw, kc, vc, [(b, pos[b]) for b in range(rows)], oshape)
        layer_s += time.perf_counter() - t0
        layers += 1
    t1 = time.perf_counter()
    logits = ogemm(ormsnorm(x, fnorm, shape.eps), head, out="f32")
    osample(logits, [[] for _ in range(rows)], [0] * rows, [OP() for _ in range(rows)])
    t2 = time.perf_counter()
    per_step = layer_s / layers * shape.n_layers + (t2 - t1)
    return {"value": round(rows / per_step, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{rows} request(s) x {layers} decoder layer(s) + final norm + LM head + sampler "
                      f"(fp64 NumPy oracle); layer time scaled to {shape.n_layers} layers",
            "seconds": round(layer_s + t2 - t1, 2)}


def run_reference(args):
    """The CPU oracle as the reference arm, on the same workload as the GPU
    arm: each step is a bounded sample -- the first min(batch, 16) requests
    of the batch (same prompt lengths) through one decoder layer, the final
    norm, the LM head and the sampler -- with the layer time scaled to the
    36-layer step."""
    ws, rank, _ = _dist()
    if rank != 0:
        return
    import torch
    from invariant_deterministic_gb300 import synth
    from oracle.gemm import gemm as ogemm
    from oracle.model import Shape, layer_step
    from oracle.rmsnorm import rmsnorm as ormsnorm
    from oracle.sampler import SamplingParams as OP, sample as osample

    cores = len(os.sched_getaffinity(0))
    oshape = Shape(d_model=4096, n_q=32, n_kv=8, head_dim=128, ffn=12288, vocab=151936, n_layers=36,
                   eps=1e-6, rope_base=1e6, qk_norm=True)
    lw = {k: synth.bits(v) for k, v in
          synth.layer_weights(4096, 32, 8, 128, 12288, 0, True, "cpu").items()}
    head = synth.bits(synth.normal_bf16((151936, 4096), 0.02, 998))
    fnorm = synth.bits(torch.ones(4096, dtype=torch.bfloat16))
    bsz = args.batch
    rows = min(bsz, 16)
    lens = replica_lengths(bsz, 0)[:rows]
    lmax = max(lens) + args.steps + args.warmup + 1
    kc = synth.bits(synth.normal_bf16((rows, lmax, 8, 128), 1.0, 1))
    vc = synth.bits(synth.normal_bf16((rows, lmax, 8, 128), 1.0, 2))
    x = synth.bits(synth.normal_bf16((rows, 4096), 1.0, 3))
    params = [OP(temperature=0.8, top_k=50, top_p=0.95, min_p=0.05, repeat_penalty=1.1,
                 repeat_last_n=64, seed=synth.SEED_REQ_BASE + b) for b in range(rows)]
    hist = [[] for _ in range(rows)]

    def one(step):
        t0 = time.perf_counter()
        y = layer_step(x, lw, kc, vc, [(b, lens[b] + step) for b in range(rows)], oshape)
        t1 = time.perf_counter()
        logits = ogemm(ormsnorm(y, fnorm, 1e-6), head, out="f32")
        osample(logits, hist, [step] * rows, params)
        t2 = time.perf_counter()
        return (t1 - t0) * 36 + (t2 - t1)

    for i in range(args.warmup):
        one(i)
    times = [one(args.warmup + i) for i in range(args.steps)]
    per_step = sum(times) / len(times)
    value = rows / per_step
    sample = (f"first {rows} of the batch's {bsz} requests x 1 Qwen3-8B-shaped decoder layer + "
              "final norm + LM head + sampler per step, fp64 NumPy oracle; layer time scaled x36")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": UNIT, "n_gpus": ws,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_step * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic: random-init weights ~N(0,0.02) bf16, prompt KV cache ~N(0,1) bf16",
        "config": {"workload": workload_name(36, bsz), "batch": bsz, "layers": 36, "split_len": 256,
                   "parallelism": f"replicas x{ws}"},
        "cpu_baseline": {"value": round(value, 5), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


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
    ap.add_argument("--no-prefill", dest="prefill", action="store_false")
    ap.add_argument("--prefill-len", type=int, default=4096)
    ap.add_argument("--prefill-chunks", default="512,4096")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    args.prefill_chunks = [int(c) for c in str(args.prefill_chunks).split(",") if c]
    if args.impl == "reference":
        run_reference(args)
    else:
        run_kinv(args)


if __name__ == "__main__":
    main()
