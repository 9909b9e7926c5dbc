#!/usr/bin/env python
"""Training-step throughput of the GB300 decoder trainer (librdt.so).

One step = forward of every block, fused final norm + LM head + cross-entropy
(forward and backward), backward of every block, the squared-sum global-norm
clip and AdamW over every fp32 master weight, on synthetic inputs already
resident in HBM. Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload q4b_full]
  python bench.py --workload q4b_nf4     # NF4-frozen block + LoRA, adapters-only step
  python bench.py --impl reference ...   # the FP64 CPU oracle on host cores

Multi-GPU (torchrun): every rank runs an independent replica of the whole
step (the path has no data-path collective); timing is the max over ranks and
`value` counts the tokens of all ranks ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import csv
import io
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "train tokens/s (fwd+bwd+clip+AdamW) at Qwen3-4B shape; % of BF16/HBM roofline"
UNIT = "tokens/s"

# DRAM traffic per tensor-core GEMM launch (dram__bytes_read.sum +
# dram__bytes_write.sum), averaged over the q4b_full step's launch mix: 36 x
# the 12 launches of one q4b_full-shaped block + the LM head's 20, each
# captured alone on that small case (the shapes are the step's), and the
# gemm.cu + api.cu sources it was measured on; reported only while they are
# unchanged.
GEMM_TRAFFIC_BYTES = 253317101
GEMM_TRAFFIC_SRC_SHA = "020eeea884ff64f1"
# The same for the 8 NF4 GEMM launches of one q4b_nf4 step.
NF4_TRAFFIC_BYTES = 75824544
NF4_TRAFFIC_SRC_SHA = "020eeea884ff64f1"


def source_sha():
    """sha256 prefix of the GEMM kernels (gemm.cu) and of the launch sequence
    that picks their shapes (api.cu): the traffic figures below hold for it."""
    import hashlib
    h = hashlib.sha256()
    for name in ("gemm.cu", "api.cu"):
        with open(os.path.join(ROOT, "resident_decoder_trainer_gb300", "csrc", name), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def traffic_if_current(nbytes, sha):
    """nbytes while gemm.cu and api.cu are the sources the counters were
    taken on, else None."""
    return nbytes if source_sha() == sha else None


def max_over_ranks(value, world, device="cpu"):
    """The maximum of a rank's value over all ranks (the value itself at N = 1):
    the slowest rank sets the job's time."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_barrier(world):
    """All ranks reach this point before any goes on (no-op at N = 1)."""
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def job_throughput(max_seconds, world, units_per_rank):
    """Whole-job throughput: the units every rank processed over the slowest
    rank's time (replicas: each rank does the same work)."""
    return world * units_per_rank / max_seconds


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["rdt", "reference"], default="rdt")
    ap.add_argument("--workload", default="q4b_full")
    ap.add_argument("--layers", type=int, default=None, help="override the layer count")
    ap.add_argument("--kernel", choices=["block", "head"], default=None,
                    help="time one block forward+backward, or the LM head + CE, alone "
                         "(small device footprint, for per-kernel numbers and ncu captures)")
    ap.add_argument("--checkpoint-segments", type=int, default=0,
                    help="activation checkpointing: hold one of N layer segments' activations "
                         "and recompute the rest in the backward (0: off)")
    ap.add_argument("--accumulation-steps", type=int, default=1,
                    help="gradient accumulation: micro-batches (of the workload's batch) per "
                         "optimizer step")
    ap.add_argument("--embedding", action="store_true",
                    help="device embedding: the step takes token ids (lookup, scatter-add "
                         "backward and the table's AdamW on the GPU)")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch the step's kernels one by one instead of replaying the "
                         "captured CUDA graph of the step")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    return ap.parse_args()


def workload_config(shape, name):
    return {
        "workload": (f"{name}: {shape.layers} Qwen3-style blocks (hidden {shape.hidden}, "
                     f"{shape.n_heads}/{shape.n_kv_heads} heads, head_dim {shape.head_dim}, "
                     f"SwiGLU {shape.intermediate}) + vocab-{shape.vocab} LM head, "
                     f"batch {shape.batch} x seq {shape.seq}"),
        "tokens_per_step": shape.tokens,
        "layers": shape.layers,
        "global_batch": shape.batch,
        "seq_len": shape.seq,
        "params": param_count(shape),
        "optimizer": "global-norm clip 1.0 + AdamW (fp32 master, m, v)",
        "l2": "inputs larger than L2: each step streams ~150 GB of weights/grads/moments",
        "parallelism": "replicas",
    }


def param_count(shape):
    """Trainable parameters of the stack: every block's seven matrices and
    four gains, the final norm gain and the LM head."""
    s = shape
    blk = ((s.q_dim + 2 * s.kv_dim) * s.hidden + s.hidden * s.q_dim
           + 3 * s.intermediate * s.hidden + 2 * s.hidden + 2 * s.head_dim)
    return s.layers * blk + s.hidden + s.vocab * s.hidden


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            pk = json.load(fh)
        return pk, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# ---------------------------------------------------------------- clocks
def start_clock_sampler(device_index):
    fd, path = tempfile.mkstemp(suffix=".csv")
    os.close(fd)
    q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    try:
        fh = open(path, "w")
        proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits",
                                 "-i", str(device_index), "-lms", "200"], stdout=fh,
                                stderr=subprocess.DEVNULL)
        return proc, fh, path
    except Exception:
        return None, None, path


def stop_clock_sampler(handle):
    proc, fh, path = handle
    if proc is None:
        return None
    proc.terminate()
    try:
        proc.wait(timeout=5)
    except Exception:
        proc.kill()
    fh.close()
    rows = []
    with open(path) as f:
        for r in csv.reader(f):
            if len(r) >= 9:
                rows.append([c.strip() for c in r])
    os.unlink(path)
    if not rows:
        return None
    sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
    mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
    load = [s for s in sm if mx and s > 0.3 * max(mx)] or sm
    return {"sm_mhz": statistics.median(load) if load else None,
            "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- CPU oracle
# The one bounded oracle sample both the cpu_baseline leg and each step of the
# reference arm time: about 11 s on 16 host cores at the q4b_full shape (a
# 5 + 20 step reference run takes about 4.5 minutes).
ORACLE_SAMPLE = dict(seqs=2, head_tokens=1024, opt_params=1 << 26)


def host_cpu():
    """Threads the oracle's BLAS uses and the host CPU's model name."""
    try:
        from threadpoolctl import threadpool_info
        cores = max(int(i.get("num_threads", 1)) for i in threadpool_info()) or os.cpu_count()
    except Exception:
        cores = os.cpu_count()
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        model = next((l.split(":", 1)[1].strip() for l in out.splitlines()
                      if l.strip().lower().startswith("model name")), None)
    except Exception:
        pass
    if not model:
        import platform
        model = platform.processor() or platform.machine()
    return cores, model


class OracleSample:
    """The FP64 oracle timed on a bounded sample of one step, scaled to the
    whole step: one block forward+backward on `seqs` of the workload's
    sequences (x layers; at most its batch), the final norm + LM head + CE
    forward and backward on
    `head_tokens` tokens (x tokens per step), and clip + AdamW on `opt_params`
    parameters (x total parameters). Inputs are drawn once (seeded)."""

    def __init__(self, shape, seqs=1, head_tokens=512, opt_params=1 << 25, seed=0):
        import numpy as np
        import torch
        from oracle import model as om
        from resident_decoder_trainer_gb300 import synth

        self.om, self.shape = om, shape
        self.s_blk = shape.replace(layers=1, batch=min(seqs, shape.batch))
        self.seq_tokens = self.s_blk.tokens
        self.head_tokens, self.opt_params = head_tokens, opt_params
        blk, x, dy = synth.make_block_inputs(self.s_blk, seed)
        self.blk = {k: om._f64(v) for k, v in blk.items()}
        self.x, self.dy = om._f64(x), om._f64(dy)
        g = torch.Generator().manual_seed(seed + 1)
        self.h = om._f64(torch.randn(head_tokens, shape.hidden, generator=g))
        self.wl = om._f64(0.02 * torch.randn(shape.vocab, shape.hidden, generator=g))
        self.gf = np.ones(shape.hidden)
        self.tg = np.random.default_rng(seed).integers(0, shape.vocab, head_tokens)
        rng = np.random.default_rng(seed)
        self.w = rng.standard_normal(opt_params)
        self.gr = rng.standard_normal(opt_params) * 1e-3
        self.m = np.zeros(opt_params)
        self.v = np.zeros(opt_params)
        self.n_params = shape.layers * sum(
            int(np.prod(sh)) for sh in synth.block_shapes(shape).values()) \
            + shape.hidden + shape.vocab * shape.hidden

    def run(self):
        om, shape = self.om, self.shape
        o = {"lr": 1e-3, "beta1": 0.9, "beta2": 0.95, "eps": 1e-8, "weight_decay": 0.1}
        t0 = time.perf_counter()
        _, cache = om.block_forward(self.blk, self.x, self.s_blk)
        om.block_backward(cache, self.dy, self.s_blk)
        t1 = time.perf_counter()
        om.head_forward_backward(self.h, self.gf, self.wl, self.tg, shape)
        t2 = time.perf_counter()
        sc, _, _ = om.clip_scale([om.squared_sum(self.gr)], 1.0)
        om.adamw(self.w, self.gr, self.m, self.v, 1, o["lr"], o["beta1"], o["beta2"], o["eps"],
                 o["weight_decay"], sc)
        t3 = time.perf_counter()
        step_s = (shape.tokens * (shape.layers * (t1 - t0) / self.seq_tokens
                                  + (t2 - t1) / self.head_tokens)
                  + (t3 - t2) * self.n_params / self.opt_params)
        cores, model = host_cpu()
        sample = (f"FP64 oracle: 1 block fwd+bwd on {self.s_blk.batch}x{self.s_blk.seq} tokens "
                  f"(x{shape.layers} layers), head+CE fwd+bwd on {self.head_tokens} tokens, "
                  f"clip+AdamW on {self.opt_params} params; scaled to {shape.tokens} tokens "
                  f"and {self.n_params} params per step")
        return {"value": round(shape.tokens / step_s, 3), "unit": UNIT, "cores": cores,
                "cpu_model": model, "kind": "oracle", "sample": sample,
                "sample_seconds": round(t3 - t0, 2)}


# ------------------------------------------------------------- GPU arm
def run_rdt(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from resident_decoder_trainer_gb300 import build, rdt, synth
    from resident_decoder_trainer_gb300.step import DecoderTrainer

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shape = synth.WORKLOADS[args.workload]
    if args.layers:
        shape = shape.replace(layers=args.layers)
    T = shape.tokens
    n_acc = max(1, args.accumulation_steps)
    tr = DecoderTrainer(shape, device=dev, checkpoint_segments=args.checkpoint_segments,
                        accumulation_steps=n_acc, embedding=args.embedding)
    tr.init_random(seed=1234 + rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321 + rank)
    nb = 4
    Ts = n_acc * T  # tokens per optimizer step
    if args.embedding:
        xs = [torch.randint(0, shape.vocab, (Ts,), device=dev, generator=gen, dtype=torch.int32)
              for _ in range(nb)]
    else:
        xs = [torch.randn(Ts, shape.hidden, device=dev, generator=gen) for _ in range(nb)]
    kw = "ids" if args.embedding else "x"
    tgs = [torch.randint(0, shape.vocab, (Ts,), device=dev, generator=gen, dtype=torch.int32)
           for _ in range(nb)]
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    first_loss = float(tr.train_step(targets=tgs[0], **{kw: xs[0]}).mean())
    gemms_per_step = (17 * shape.layers + 3) * n_acc  # 12 per layer, 5 more when recomputed
    use_graph = not args.no_graph
    if use_graph:
        # capture the step once (the first call captures, then replays)
        lc0 = rdt.launch_count()
        tr.train_step_graph(targets=tgs[1 % nb], **{kw: xs[1 % nb]})
        launches_per_step = rdt.launch_count() - lc0
        step_fn, first_warm = tr.train_step_graph, 2
    else:
        timer = rdt.GemmTimer(gemms_per_step * args.steps)
        step_fn, first_warm = tr.train_step, 1
    for i in range(first_warm, args.warmup):
        step_fn(targets=tgs[i % nb], **{kw: xs[i % nb]})
    barrier()
    clk = start_clock_sampler(local_rank)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = rdt.launch_count()
    if use_graph:
        e0.record(stream)
        for i in range(args.steps):
            step_fn(targets=tgs[i % nb], **{kw: xs[i % nb]})
        e1.record(stream)
        barrier()
        launches = launches_per_step * args.steps
        # per-GEMM durations: events recorded inside a graph cannot be timed,
        # so the same step runs once more with its kernels launched one by one
        timer = rdt.GemmTimer(gemms_per_step)
        with timer:
            tr.train_step(targets=tgs[0], **{kw: xs[0]})
        torch.cuda.synchronize()
    else:
        with timer:
            e0.record(stream)
            for i in range(args.steps):
                step_fn(targets=tgs[i % nb], **{kw: xs[i % nb]})
            e1.record(stream)
            barrier()
        launches = rdt.launch_count() - l0
    clocks = stop_clock_sampler(clk)
    dev_ms = e0.elapsed_time(e1)
    last_loss = float(tr.loss_partials.mean())
    max_ms = max_over_ranks(dev_ms, world, dev)
    value = job_throughput(max_ms / 1e3, world, Ts * args.steps)

    res = timer.results()
    gemm_flops = sum(f for f, _ in res)
    gemm_ms = sum(ms for _, ms in res)
    peaks, peak_kind = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops"))
    achieved = gemm_flops / (gemm_ms / 1e3) / 1e12 if gemm_ms > 0 else None
    n_launch = len(res)
    traffic = traffic_if_current(GEMM_TRAFFIC_BYTES, GEMM_TRAFFIC_SRC_SHA)
    roofline = {
        "kernel": "gemm_kernel / gemm2_kernel (tcgen05 BF16 single-CTA 128x192/256 and CTA-pair 256x256 tiles, TMEM fp32 accumulators, TMA)",
        "bound": "tensor", "achieved": round(achieved, 1) if achieved else None,
        "peak": peak_tf, "unit": "TFLOP/s",
        "frac": round(achieved / peak_tf, 4) if achieved else None,
        "peak_source": f"bf16_tflops_sustained of {peak_kind}",
        "traffic": traffic,
        "launches_timed": n_launch,
        "flops_per_launch": gemm_flops / max(n_launch, 1),
        "ms_per_launch": gemm_ms / max(n_launch, 1),
        "gemm_share_of_step": round(gemm_ms / (max_ms * (1 if use_graph else args.steps)
                                               / args.steps), 4) if max_ms else None,
    }
    step_flops = algorithmic_flops(shape) * n_acc
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic (device-generated N(0,1) hidden states, uniform ids;"
                                  " N(0,0.02) random-init weights)",
        "config": workload_config(shape, args.workload),
        "roofline": roofline,
        "step_tflops": round(step_flops / (max_ms / args.steps / 1e3) / 1e12, 1),
        "gpu_launches": int(launches),
        "clocks": clocks,
        "loss_first_step": round(first_loss, 5), "loss_last_step": round(last_loss, 5),
        "launch": "one CUDA graph replay per step" if use_graph else "eager kernel launches",
    }
    out["config"]["algorithmic_tflop_per_step"] = round(step_flops / 1e12, 2)
    out["config"]["activation_gb_held"] = round(tr.saved.numel() / 1e9, 2)
    if args.embedding:
        out["config"]["embedding"] = ("device lookup + deterministic scatter-add backward + "
                                      "the table's own AdamW")
        out["config"]["params"] = param_count(shape) + shape.vocab * shape.hidden
        out["data"] = ("synthetic (device-generated uniform token ids and targets; N(0,0.02) "
                       "random-init weights, N(0,1) embedding table)")
    if n_acc > 1:
        out["config"]["tokens_per_step"] = Ts
        out["config"]["global_batch"] = shape.batch * n_acc
        out["config"]["accumulation_steps"] = n_acc
    if args.checkpoint_segments:
        out["config"]["activation_checkpointing"] = {
            "segments": args.checkpoint_segments, "layers_per_segment": tr.segment_size,
            "activation_gb_without": round(shape.layers * tr.saved_bytes / 1e9, 2)}

    if not args.no_e2e:
        out["e2e"] = run_e2e(tr, shape, args, dev, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = OracleSample(shape, **ORACLE_SAMPLE).run()
    return out


def run_e2e(tr, shape, args, dev, world):
    """Same metric through the public API with HOST buffers: every step copies
    its inputs from pinned host memory and reads its loss partials back."""
    import torch
    T = shape.tokens * tr.accumulation_steps
    if tr.embedding:  # the inputs are token ids
        xh = torch.randint(0, shape.vocab, (T,), dtype=torch.int32).pin_memory()
    else:
        xh = torch.randn(T, shape.hidden).pin_memory()
    th = torch.randint(0, shape.vocab, (T,), dtype=torch.int32).pin_memory()
    lh = torch.empty(T, dtype=torch.float32).pin_memory()
    xd = torch.empty(xh.shape, dtype=xh.dtype, device=dev)
    td = torch.empty(T, dtype=torch.int32, device=dev)
    kw = "ids" if tr.embedding else "x"
    # events around the copies (on the step's stream) show their share of the
    # wall time; they do not change what is timed
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    rank_barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(args.steps):
        ev[i][0].record()
        xd.copy_(xh, non_blocking=True)
        td.copy_(th, non_blocking=True)
        ev[i][1].record()
        loss = (tr.train_step if args.no_graph else tr.train_step_graph)(targets=td,
                                                                          **{kw: xd})
        ev[i][2].record()
        lh.copy_(loss, non_blocking=True)
        ev[i][3].record()
        torch.cuda.current_stream().synchronize()  # the caller reads this step's loss
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    dt = max_over_ranks(wall, world, dev)
    h2d = statistics.mean(e[0].elapsed_time(e[1]) for e in ev)
    d2h = statistics.mean(e[2].elapsed_time(e[3]) for e in ev)
    return {"value": round(job_throughput(dt, world, T * args.steps), 1), "unit": UNIT,
            "h2d_bytes_per_step": xh.numel() * 4 + th.numel() * 4,
            "d2h_bytes_per_step": lh.numel() * 4,
            "wall_ms_per_step": round(wall * 1e3 / args.steps, 3),
            "h2d_ms_per_step": round(h2d, 4), "d2h_ms_per_step": round(d2h, 4)}


def algorithmic_flops(shape):
    """Dense-contraction FLOPs of one step: 6 x params x tokens for every
    projection and the LM head, plus 6 causal attention matmuls
    (2 nh d (S+1)/2 per token each) per layer."""
    s = shape
    blk = (s.q_dim + 2 * s.kv_dim) * s.hidden + s.hidden * s.q_dim + 3 * s.intermediate * s.hidden
    proj = 6.0 * (s.layers * blk + s.vocab * s.hidden) * s.tokens
    attn = s.layers * 6 * 2.0 * s.n_heads * s.head_dim * (s.seq + 1) / 2 * s.tokens
    return proj + attn


# ------------------------------------------------- NF4 + LoRA workload
NF4_WORKLOADS = ("q4b_nf4",)


def nf4_workload_config(shape, name, rank, alpha):
    return {
        "workload": (f"{name}: one Qwen3-style block (hidden {shape.hidden}, {shape.n_heads}/"
                     f"{shape.n_kv_heads} heads, head_dim {shape.head_dim}, SwiGLU "
                     f"{shape.intermediate}) with frozen NF4 projections (64-weight blocks, "
                     f"fp32 scales) and LoRA rank {rank} / alpha {alpha:g} on all seven; "
                     f"batch {shape.batch} x seq {shape.seq}"),
        "tokens_per_step": shape.tokens,
        "layers": shape.layers,
        "global_batch": shape.batch,
        "seq_len": shape.seq,
        "params": rank * sum(o + i for o, i in (
            (shape.q_dim, shape.hidden), (shape.kv_dim, shape.hidden),
            (shape.kv_dim, shape.hidden), (shape.hidden, shape.q_dim),
            (shape.intermediate, shape.hidden), (shape.intermediate, shape.hidden),
            (shape.hidden, shape.intermediate))),
        "optimizer": "global-norm clip 1.0 + AdamW over the adapters (fp32 master, m, v)",
        "l2": "flushed: a 256 MB buffer is written between timed steps",
        "parallelism": "replicas",
    }


def nf4_algorithmic_flops(shape, rank):
    """Dense-contraction FLOPs of one adapters-only step: forward and input
    gradient through the seven frozen projections (4 x params x tokens; no
    weight gradient), the six causal attention matmuls, and the LoRA terms
    (6 T r (in + out) per projection: U, its tail product, dU, the tail of
    the input gradient, dA and dB)."""
    from resident_decoder_trainer_gb300 import synth
    s = shape
    shp = synth.block_shapes(s)
    proj = sum(shp[n][0] * shp[n][1] for n in synth.NF4_PROJECTIONS)
    lora = sum(shp[n][0] + shp[n][1] for n in synth.NF4_PROJECTIONS)
    attn = 6 * 2.0 * s.n_heads * s.head_dim * (s.seq + 1) / 2 * s.tokens
    return 4.0 * proj * s.tokens + 6.0 * rank * lora * s.tokens + attn


class Nf4OracleSample:
    """The FP64 NF4 + LoRA oracle timed on a bounded sample of one step: the
    block forward+backward on `seqs` of the workload's sequences (at most its
    batch; scaled to the step's tokens) plus the adapters' clip + AdamW (the
    full adapter set)."""

    def __init__(self, shape, rank, alpha, seqs=1, seed=0):
        import numpy as np
        from oracle import model as om
        from oracle import nf4 as on
        from resident_decoder_trainer_gb300 import synth
        self.om, self.on, self.np = om, on, np
        self.shape, self.rank, self.alpha = shape, rank, alpha
        self.s_blk = shape.replace(layers=1, batch=min(seqs, shape.batch))
        self.seq_tokens = self.s_blk.tokens
        base, gains, lora, x, dy = synth.make_nf4_inputs(self.s_blk, seed=seed, rank=rank,
                                                         b_std=0.02)
        shp = synth.block_shapes(self.s_blk)
        self.base = {k: on.nf4_dequantize(p.numpy(), a.numpy(), *shp[k])
                     for k, (p, a) in base.items()}
        self.gains = {k: v.numpy().astype(np.float64) for k, v in gains.items()}
        self.lora = {k: v.numpy().astype(np.float64) for k, v in lora.items()}
        self.x, self.dy = om._f64(x), om._f64(dy)

    def run(self):
        import time as _t
        from resident_decoder_trainer_gb300 import synth
        t0 = _t.perf_counter()
        self.on.lora_step(self.base, self.gains, self.lora, self.x, self.dy, self.s_blk,
                          self.rank, self.alpha, synth.OPTIM)
        dt = _t.perf_counter() - t0
        step_s = dt * self.shape.tokens / self.seq_tokens
        cores, model = host_cpu()
        sample = (f"FP64 NF4+LoRA oracle: block fwd+bwd + adapter clip+AdamW on "
                  f"{self.s_blk.batch}x{self.s_blk.seq} tokens, scaled to {self.shape.tokens} "
                  "tokens per step")
        return {"value": round(self.shape.tokens / step_s, 3), "unit": UNIT, "cores": cores,
                "cpu_model": model, "kind": "oracle", "sample": sample,
                "sample_seconds": round(dt, 2)}


def run_nf4(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist
    from resident_decoder_trainer_gb300 import build, rdt, synth
    from resident_decoder_trainer_gb300.nf4_step import Nf4LoraTrainer

    build.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    shape = synth.WORKLOADS[args.workload]
    T = shape.tokens
    tr = Nf4LoraTrainer(shape, device=dev)
    tr.init_random(seed=1234 + rank)
    gen = torch.Generator(device=dev)
    gen.manual_seed(4321 + rank)
    nb = 4
    xs = [torch.randn(T, shape.hidden, device=dev, generator=gen) for _ in range(nb)]
    dys = [1e-3 * torch.randn(T, shape.hidden, device=dev, generator=gen) for _ in range(nb)]
    # the step's working set (~1.5 GB) would otherwise sit in L2 between steps
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()

    use_graph = not args.no_graph
    tr.train_step(xs[0], dys[0])
    if use_graph:
        lc0 = rdt.launch_count()
        tr.train_step_graph(xs[1 % nb], dys[1 % nb])  # captures, then replays
        launches_per_step = rdt.launch_count() - lc0
    for i in range(2 if use_graph else 1, args.warmup):
        (tr.train_step_graph if use_graph else tr.train_step)(xs[i % nb], dys[i % nb])
    timer = rdt.GemmTimer(32 * (1 if use_graph else args.steps))
    barrier()
    clk = start_clock_sampler(local_rank)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(args.steps)]
    l0 = rdt.launch_count()
    if use_graph:
        for i in range(args.steps):
            # inputs staged and L2 flushed outside the timed events
            tr.x_stage.copy_(xs[i % nb])
            tr.dy_stage.copy_(dys[i % nb])
            flush.fill_(i & 0xFF)
            evs[i][0].record(stream)
            tr.train_step_graph()
            evs[i][1].record(stream)
        barrier()
        launches = launches_per_step * args.steps
        with timer:  # per-GEMM durations on one eager step (graph events cannot be timed)
            tr.train_step(xs[0], dys[0])
        torch.cuda.synchronize()
    else:
        with timer:
            for i in range(args.steps):
                flush.fill_(i & 0xFF)  # outside the timed events: evicts the previous step
                evs[i][0].record(stream)
                tr.train_step(xs[i % nb], dys[i % nb])
                evs[i][1].record(stream)
            barrier()
        launches = rdt.launch_count() - l0
    clocks = stop_clock_sampler(clk)
    dev_ms = sum(a.elapsed_time(b) for a, b in evs)
    max_ms = max_over_ranks(dev_ms, world, dev)
    value = job_throughput(max_ms / 1e3, world, T * args.steps)

    res = timer.results(with_kind=True)
    nf4 = [(f, ms) for f, ms, k in res if k == "nf4"]
    other = [(f, ms) for f, ms, k in res if k != "nf4"]
    nf4_flops, nf4_ms = sum(f for f, _ in nf4), sum(ms for _, ms in nf4)
    peaks, peak_kind = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained") or peaks.get("bf16_tflops"))
    achieved = nf4_flops / (nf4_ms / 1e3) / 1e12 if nf4_ms > 0 else None
    roofline = {
        "kernel": "gemm2_nf4_kernel (tcgen05 BF16 CTA pairs, 256x256 tiles, B decoded from "
                  "4-bit NF4 codes + per-64 fp32 scales into shared memory by two groups of "
                  "four decode warps on alternate k-blocks, LoRA term as a bf16 tail k-block)",
        "bound": "tensor", "achieved": round(achieved, 1) if achieved else None,
        "peak": peak_tf, "unit": "TFLOP/s",
        "frac": round(achieved / peak_tf, 4) if achieved else None,
        "peak_source": f"bf16_tflops_sustained of {peak_kind}",
        "traffic": traffic_if_current(NF4_TRAFFIC_BYTES, NF4_TRAFFIC_SRC_SHA),
        "launches_timed": len(nf4),
        "flops_per_launch": nf4_flops / max(len(nf4), 1),
        "ms_per_launch": nf4_ms / max(len(nf4), 1),
        "nf4_gemm_share_of_step": round(nf4_ms / (max_ms / args.steps * (
            1 if use_graph else args.steps)), 4) if max_ms else None,
        "adapter_gemm_share_of_step": round(sum(ms for _, ms in other) / (
            max_ms / args.steps * (1 if use_graph else args.steps)), 4) if max_ms else None,
    }
    step_flops = nf4_algorithmic_flops(shape, tr.rank)
    out = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16 (NF4-decoded weights)",
        "data": "synthetic (device-generated N(0,1) inputs, N(0,1e-3) upstream gradients, "
                "uniform NF4 codes, 3|N(0,0.02)| scales, A ~ N(0,0.02), B = 0)",
        "config": nf4_workload_config(shape, args.workload, tr.rank, tr.alpha),
        "roofline": roofline,
        "step_tflops": round(step_flops / (max_ms / args.steps / 1e3) / 1e12, 1),
        "gpu_launches": int(launches),
        "clocks": clocks,
        "launch": "one CUDA graph replay per step" if use_graph else "eager kernel launches",
    }
    out["config"]["algorithmic_tflop_per_step"] = round(step_flops / 1e12, 3)
    if not args.no_e2e:
        xh = [x.cpu().pin_memory() for x in xs[:2]]
        dyh = [d.cpu().pin_memory() for d in dys[:2]]
        sq_h = torch.empty(1, dtype=torch.float64).pin_memory()
        xd, dyd = torch.empty_like(xs[0]), torch.empty_like(dys[0])
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
        rank_barrier(world)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        for i in range(args.steps):
            ev[i][0].record()
            xd.copy_(xh[i % 2], non_blocking=True)
            dyd.copy_(dyh[i % 2], non_blocking=True)
            ev[i][1].record()
            (tr.train_step_graph if use_graph else tr.train_step)(xd, dyd)
            ev[i][2].record()
            sq_h.copy_(tr.sumsq, non_blocking=True)
            ev[i][3].record()
            torch.cuda.current_stream().synchronize()  # the caller reads this step's result
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        dt = max_over_ranks(wall, world, dev)
        out["e2e"] = {"value": round(job_throughput(dt, world, T * args.steps), 1), "unit": UNIT,
                      "h2d_bytes_per_step": 2 * T * shape.hidden * 4,
                      "d2h_bytes_per_step": 8,
                      "wall_ms_per_step": round(wall * 1e3 / args.steps, 3),
                      "h2d_ms_per_step": round(statistics.mean(
                          e[0].elapsed_time(e[1]) for e in ev), 4),
                      "d2h_ms_per_step": round(statistics.mean(
                          e[2].elapsed_time(e[3]) for e in ev), 4)}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        out["cpu_baseline"] = Nf4OracleSample(shape, tr.rank, tr.alpha).run()
    return out


# ---------------------------------------------------------- kernel probes
def run_probe(args):
    """One block forward+backward (or the fused LM head + CE) of the workload's
    shapes on device-resident random inputs, timed with CUDA events."""
    import torch
    from resident_decoder_trainer_gb300 import build, rdt, synth
    build.build()
    shape = synth.WORKLOADS[args.workload]
    cfg = rdt.Config.from_shape(shape)
    dev = torch.device("cuda", 0)
    gen = torch.Generator(device=dev)
    gen.manual_seed(7)
    T = shape.tokens
    sq = torch.zeros(1, dtype=torch.float64, device=dev)
    if args.kernel == "block":
        n = rdt.block_param_count(cfg)
        w = torch.empty(n, device=dev)
        for name, (o, c) in rdt.block_param_offsets(cfg).items():
            if name.startswith("g_"):
                w[o:o + c].fill_(1.0)
            else:
                w[o:o + c].normal_(0, 0.02, generator=gen)
        wb = torch.empty(n, dtype=torch.bfloat16, device=dev)
        rdt.cast_bf16(w, wb)
        saved = torch.empty(rdt.block_saved_bytes(cfg, shape.batch, shape.seq), dtype=torch.uint8,
                            device=dev)
        ws = torch.empty(rdt.block_workspace_bytes(cfg, shape.batch, shape.seq),
                         dtype=torch.uint8, device=dev)
        x = torch.randn(T, shape.hidden, device=dev, generator=gen)
        dy = 1e-3 * torch.randn(T, shape.hidden, device=dev, generator=gen)
        y, dx = torch.empty_like(x), torch.empty_like(x)
        grads = torch.empty(n, device=dev)

        def run():
            rdt.block_forward(cfg, shape.batch, shape.seq, w, wb, x, y, saved, ws)
            rdt.block_backward(cfg, shape.batch, shape.seq, w, wb, x, saved, dy, dx, grads, ws,
                               grad_sq=sq)
        s1 = shape.replace(layers=1, vocab=0)
        flops = algorithmic_flops(s1)
        what = "one block forward+backward"
    else:
        h = torch.randn(T, shape.hidden, device=dev, generator=gen)
        gf = torch.ones(shape.hidden, device=dev)
        wl = (0.02 * torch.randn(shape.vocab, shape.hidden, device=dev, generator=gen)).to(
            torch.bfloat16)
        tg = torch.randint(0, shape.vocab, (T,), device=dev, generator=gen, dtype=torch.int32)
        ws = torch.empty(rdt.head_workspace_bytes(cfg, T), dtype=torch.uint8, device=dev)
        loss = torch.empty(T, device=dev)
        dh, dgf = torch.empty_like(h), torch.empty_like(gf)
        dwl = torch.empty(shape.vocab, shape.hidden, device=dev)

        def run():
            rdt.fused_cross_entropy(cfg, T, h, gf, wl, tg, 1.0 / T, loss, dh, dgf, dwl, ws,
                                    grad_sq=sq)
        flops = 6.0 * shape.vocab * shape.hidden * T
        what = "final RMSNorm + LM head + cross-entropy, forward+backward"
    for _ in range(args.warmup):
        run()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(args.steps):
        run()
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / args.steps
    return {"probe": args.kernel, "what": what, "workload": args.workload, "tokens": T,
            "ms": round(ms, 4), "tokens_per_s": round(T / ms * 1e3, 1),
            "algorithmic_tflops": round(flops / ms / 1e9, 1), "steps": args.steps,
            "warmup": args.warmup}


# ------------------------------------------------------------ reference
def run_reference_nf4(args, world):
    from resident_decoder_trainer_gb300 import synth
    shape = synth.WORKLOADS[args.workload]
    rank_, alpha = synth.LORA["rank"], synth.LORA["alpha"]
    sampler = Nf4OracleSample(shape, rank_, alpha)
    samples = []
    for i in range(args.warmup + args.steps):
        r = sampler.run()
        if i >= args.warmup:
            samples.append(r)
    value = statistics.median(r["value"] for r in samples)
    cpu = dict(samples[-1])
    cpu["value"] = value
    sample_ms = statistics.mean(r["sample_seconds"] for r in samples) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sample_ms, 1),
        "step": ("one bounded oracle sample (cpu_baseline.sample); value scales it to the "
                 "whole step"),
        "whole_step_s_extrapolated": round(shape.tokens / value, 1),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": nf4_workload_config(shape, args.workload, rank_, alpha),
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference(args, rank, world):
    from resident_decoder_trainer_gb300 import synth
    if args.workload in NF4_WORKLOADS:
        return run_reference_nf4(args, world)
    shape = synth.WORKLOADS[args.workload]
    if args.layers:
        shape = shape.replace(layers=args.layers)
    sampler = OracleSample(shape, **ORACLE_SAMPLE)
    samples = []
    for i in range(args.warmup + args.steps):
        r = sampler.run()
        if i >= args.warmup:
            samples.append(r)
    vals = [r["value"] for r in samples]
    value = statistics.median(vals)
    cpu = dict(samples[-1])
    cpu["value"] = value
    # a reference step is one bounded oracle sample; its wall time is what ran
    sample_ms = statistics.mean(r["sample_seconds"] for r in samples) * 1e3
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sample_ms, 1),
        "step": ("one bounded oracle sample (cpu_baseline.sample); value scales it to the "
                 "whole step"),
        "whole_step_s_extrapolated": round(shape.tokens / value, 1),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(shape, args.workload),
        "cpu_baseline": cpu,
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return 0
        print(json.dumps(run_reference(args, rank, world)), flush=True)
        return 0
    if args.kernel:
        print(json.dumps(run_probe(args)), flush=True)
        return 0
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.workload in NF4_WORKLOADS:
        out = run_nf4(args, rank, world, local_rank)
    else:
        out = run_rdt(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
