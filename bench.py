"""Decode throughput of the batch-1 Llama decode pass on GB300.

Workload: Llama-3.2-1B-shaped model with Q8_0 weights (16 layers, d 2048,
32/8 heads of 64, FFN 8192, vocab 128256, tied output, RoPE base 500000 with
unit frequency factors), seeded synthetic weights, the F16 KV cache pre-filled
with 4095 seeded rows, one decode step at pos 4095 (context 4096) per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One JSON line on rank 0.  ``value`` is device-timed decode tok/s (CUDA events
on the library's stream, inputs resident in HBM; the step reads 1.45 GB, far
more than the 129 MB L2, so no flush is needed).  ``e2e`` is the same metric
through the synchronous C-ABI call with pinned host buffers (token in, argmax
and logits out).  ``roofline`` relates the step kernel's algorithmic bytes to
the measured HBM copy bandwidth.  With N > 1 every rank runs an independent
replica (a batch-1 step does not shard); ``value`` sums the ranks.
``--impl reference`` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "decode tok/s @batch1 (Llama-3.2-1B-shape Q8_0, ctx 4k); % HBM roofline"
POS = 4095
CFG = synth.LLAMA1B_Q8
# decode workloads: (model, label); the headline is the 1B shape at pos 4095
DECODE_MODELS = {"llama1b_q8": (synth.LLAMA1B_Q8, "llama-3.2-1b-shape q8_0"),
                 "llama7b_q8": (synth.LLAMA7B_Q8, "llama-2-7b-shape q8_0")}
DTYPE = "q8_0 weights x 24-bit block fixed-point activations (dp4a), f32 accumulate"
DTYPE_LLAMACPP = "q8_0 weights x q8_0-quantized activations (dp4a), f32 accumulate; f16 attention probabilities"
KERNEL_SOURCES = ["llama_decode_forward_gb300/csrc/decode_step.cu", "llama_decode_forward_gb300/csrc/llm_internal.cuh"]


# ------------------------------------------------------- byte accounting --
def weight_bytes(cfg, n_elems: int) -> int:
    return {synth.F32: 4 * n_elems, synth.F16: 2 * n_elems, synth.Q8_0: n_elems // 32 * 34}[cfg.wtype]


def matrix_elems(cfg) -> tuple[int, int]:
    """(elements of the layer matrices, elements of the logits matrix)."""
    d, q, kv, f = cfg.dim, cfg.q_dim, cfg.kv_dim, cfg.ffn_dim
    per_layer = d * q + 2 * d * kv + q * d + 3 * d * f
    return cfg.n_layers * per_layer, cfg.vocab * d


def algorithmic_bytes(cfg, pos: int) -> int:
    """Bytes one decode step must move: every matrix once (the logits matrix is
    the embedding when tied), the F32 norm gains and biases, and the F16 K/V
    rows 0..pos of every layer."""
    layers, logits = matrix_elems(cfg)
    b = weight_bytes(cfg, layers) + weight_bytes(cfg, logits)
    b += 4 * (2 * cfg.n_layers + 1) * cfg.dim
    if cfg.bias:
        b += 4 * cfg.n_layers * (cfg.q_dim + 2 * cfg.kv_dim)
    b += (pos + 1) * cfg.n_layers * 2 * cfg.kv_dim * 2
    return b


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def kernel_hash() -> str:
    h = hashlib.sha256()
    for s in KERNEL_SOURCES:
        with open(os.path.join(ROOT, s), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def stored_traffic():
    """Per-launch DRAM bytes from the committed ncu summary, if it was taken
    on the current kernel source."""
    p = os.path.join(ROOT, "profiles", "decode_step_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("kernel_hash") != kernel_hash() or d.get("pos") != POS:
        return None
    return d.get("dram_bytes_per_launch")


# ------------------------------------------------------------ clocks --
class ClockSampler:
    def __init__(self, device_uuid: str | None):
        self.proc = None
        self.path = None
        q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
        cmd = ["nvidia-smi", f"--query-gpu={q}", "--format=csv,noheader,nounits", "-lms", "100"]
        if device_uuid:
            cmd += ["-i", device_uuid]
        try:
            import tempfile
            self.path = tempfile.mktemp(suffix=".csv")
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict | None:
        if not self.proc:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------ ranks --
def max_over_ranks(x: float, world: int, device) -> float:
    """The largest of every rank's x: the job lasts as long as its slowest
    rank.  One all-reduce on the process group (NCCL on the GPU machine, gloo in
    the CPU tests)."""
    if world <= 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, seconds: float) -> float:
    """Tokens per second of the whole job: each of the `world` ranks decodes
    `steps` tokens of its own replica, and `seconds` is the slowest rank's time."""
    return world * steps / seconds


# --------------------------------------------------------- CPU baseline --
def cpu_oracle_sample(W, tok: int, budget_s: float = 12.0, min_steps: int = 1, max_steps: int | None = None,
                      cfg=None, pos: int = POS, threads: int = 1):
    """The oracle on the same workload: decode steps at `pos` after the same
    pre-filled rows, as many as fit in the budget; on one thread, or with
    `threads` > 1 its row-split variant (bitwise the same results)."""
    import oracle
    cfg = cfg or CFG
    ora = oracle.OracleModel(cfg, W, max_seq=pos + 1, llamacpp_rounding=bool(getattr(cfg, "numerics", 0)))
    for l in range(cfg.n_layers):
        for which in (0, 1):
            if pos:
                ora.set_kv_rows_f16(l, which, synth.kv_rows(cfg, l, which, pos))
    oracle.set_threads(threads)
    try:
        n, t0 = 0, time.perf_counter()
        while True:
            ora.forward(tok, pos)
            n += 1
            el = time.perf_counter() - t0
            if (n >= min_steps and el >= budget_s) or (max_steps and n >= max_steps):
                break
    finally:
        oracle.set_threads(1)
        ora.close()
    return n, el


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    W = synth.make_weights(CFG)
    tok = int(synth.prompt(CFG, 1)[0])
    warm = min(args.warmup, 1)
    if warm:
        cpu_oracle_sample(W, tok, budget_s=0.0, min_steps=warm, max_steps=warm)
    n, el = cpu_oracle_sample(W, tok, budget_s=min(180.0, 10.0 * max(1, args.steps)), min_steps=1,
                              max_steps=args.steps)
    v = n / el
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tok/s", "n_gpus": args.gpus, "steps": n,
            "warmup": warm, "ms_per_step": 1000.0 * el / n, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "q8_0 weights x f32 activations, f32 accumulate",
            "data": "synthetic (seeded random Q8_0 weights and KV rows)",
            "config": {"workload": "llama-3.2-1b-shape q8_0 decode, batch 1, step at pos 4095 (ctx 4096)",
                       "pos": POS, "implementation": "CPU oracle (plain C, single thread)"},
            "cpu_baseline": {"value": v, "unit": "tok/s", "cores": 1, "kind": "oracle",
                             "sample": f"{n} full decode steps at pos 4095, 1 thread"},
            "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------- ours --
def percentiles(xs) -> dict:
    """Median and the 10th / 90th percentiles of per-launch times (ms)."""
    a = np.sort(np.asarray(xs, dtype=np.float64))
    q = lambda f: float(np.quantile(a, f))
    return {"median": q(0.5), "p10": q(0.1), "p90": q(0.9), "n": int(a.size)}


def run_ours(args):
    import torch
    import torch.distributed as dist
    import llama_decode_forward_gb300 as L

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.cuda.current_device()

    cfg, label = DECODE_MODELS[args.model]
    pos = POS if args.pos is None else args.pos
    lc = args.numerics == "llamacpp"
    headline = args.model == "llama1b_q8" and pos == POS and not lc
    cfg = cfg.scaled(max_seq=max(cfg.max_seq if headline else 0, pos + 1), numerics=int(lc))
    W = synth.make_weights(cfg)
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        dec = L.Decoder(cfg, W, stream=stream.cuda_stream)
        for l in range(cfg.n_layers):
            k, v = dec.kv_tensors(l)
            for which, t in ((0, k), (1, v)):
                if pos:
                    rows = synth.kv_rows(cfg, l, which, pos)
                    t[:pos].copy_(torch.from_numpy(rows.view(np.int16)).to("cuda"))
    torch.cuda.synchronize()
    tok = int(synth.prompt(cfg, 1)[0])
    token_dev = torch.tensor([tok], dtype=torch.int32, device="cuda")
    argmax_dev = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        L.llm_decode_step_async(dec.h, token_dev, pos, argmax_dev)

    for _ in range(max(args.warmup, 3)):
        step()
    L.llm_sync(dec.h)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()

    uuid = None
    try:
        uuid = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        pass
    clocks = ClockSampler(uuid)
    time.sleep(0.3)
    launches0 = L.llm_launch_count(dec.h)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    t_start.record(stream)
    for i in range(args.steps):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    t_end.record(stream)
    torch.cuda.synchronize()
    launches = L.llm_launch_count(dec.h) - launches0
    L.llm_sync(dec.h)
    clk = clocks.stop()
    total_ms = t_start.elapsed_time(t_end)
    per_launch = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total_ms = max_over_ranks(total_ms, world, "cuda")
    value = job_throughput(world, args.steps, total_ms / 1000.0)

    # end to end through the synchronous C-ABI call, pinned host buffers
    logits_pin = torch.empty(cfg.vocab, dtype=torch.float32, pin_memory=True)
    logits_np = logits_pin.numpy()
    for _ in range(max(args.warmup, 3)):
        L.llm_decode_step(dec.h, tok, pos, logits_np)
    if world > 1:
        dist.barrier()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        L.llm_decode_step(dec.h, tok, pos, logits_np)
    e2e_s = time.perf_counter() - t0
    e2e_s = max_over_ranks(e2e_s, world, "cuda")
    e2e = job_throughput(world, args.steps, e2e_s)

    nbytes = algorithmic_bytes(cfg, pos)
    kern_ms = statistics.mean(per_launch)
    peaks = measured_peaks()
    achieved = nbytes / (kern_ms / 1000.0) / 1e9
    traffic = stored_traffic() if headline else None
    pct = percentiles(per_launch)
    line = {
        "metric": METRIC if headline else (f"decode tok/s @batch1 ({label}, step at pos {pos}"
                                           f"{', llama.cpp rounding' if lc else ''}); % HBM roofline"),
        "value": value, "unit": "tok/s", "n_gpus": world, "steps": args.steps,
        "warmup": max(args.warmup, 3), "ms_per_step": total_ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": DTYPE_LLAMACPP if lc else DTYPE,
        "data": "synthetic (seeded random Q8_0 weights and KV rows)",
        "config": {"workload": f"{label} decode, batch 1, step at pos {pos} (ctx {pos + 1})"
                               + (", llama.cpp rounding" if lc else ""),
                   "n_layers": cfg.n_layers, "dim": cfg.dim, "vocab": cfg.vocab, "pos": pos,
                   "bytes_per_step": nbytes,
                   "l2": f"working set {nbytes / 1e9:.2f} GB > 129 MB L2; no flush",
                   "parallelism": f"replicas x{world}"},
        "launch_ms": pct,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": achieved / peaks["hbm_gbs"], "traffic": traffic,
                     "kernel": f"decode_step_kernel<Q8_0{', llama.cpp rounding' if lc else ''}> (whole step, one launch)",
                     "peak_source": peaks["source"] + " (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)",
                     "frac_of_8tbs_nominal": achieved / 8000.0,
                     "frac_at_median_launch": nbytes / (pct["median"] / 1000.0) / 1e9 / peaks["hbm_gbs"]},
        "e2e": {"value": e2e, "unit": "tok/s", "h2d_bytes_per_step": 4, "d2h_bytes_per_step": 4 + 4 + 4 * cfg.vocab},
        "gpu_launches": launches,
        "clocks": clk,
    }
    if rank == 0 and not args.no_cpu_baseline:
        n, el = cpu_oracle_sample(W, tok, budget_s=args.cpu_budget, cfg=cfg, pos=pos)
        line["cpu_baseline"] = {"value": n / el, "unit": "tok/s", "cores": 1, "kind": "oracle",
                                "sample": f"{n} full decode steps at pos {pos} of the same model, 1 thread, {el:.1f} s"}
        cores = os.cpu_count() or 1
        n, el = cpu_oracle_sample(W, tok, budget_s=args.cpu_budget, cfg=cfg, pos=pos, threads=cores)
        line["cpu_baseline_all_cores"] = {
            "value": n / el, "unit": "tok/s", "cores": cores, "kind": "oracle (row-split over the host cores)",
            "sample": f"{n} full decode steps at pos {pos} of the same model, {cores} threads, {el:.1f} s "
                      "(each output element computed by one thread: bitwise the single-thread result)"}
    dec.close()
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(line))
    return 0


# ------------------------------------------------------------- prefill --
PREFILL_CFGS = {"f16": synth.QWEN2_F16, "q8_0": synth.LLAMA1B_Q8}
PREFILL_N = 512


def prefill_flops(cfg, n: int) -> float:
    """FLOPs of one n-token prefill from position 0: the layer GEMMs (2 per
    multiply-add), causal attention (q.k and p.v over positions 0..i for every
    row i), and the last row's logits."""
    layers, _ = matrix_elems(cfg)
    gemm = 2.0 * layers * n
    attn = cfg.n_layers * cfg.n_heads * cfg.head_dim * 4.0 * (n * (n + 1) / 2)
    logits = 2.0 * cfg.vocab * cfg.dim
    return gemm + attn + logits


def run_prefill(args):
    """Optional line (not the headline): a 1B-shape model's 512-token batched
    prefill (the Qwen2-style F16 model, or Llama 3.2 Q8_0 whose quants are
    expanded to F16 tile by tile inside each GEMM, or with --prefill-f16-copy
    read from the handle's F16 copy of the layer matrices), tokens per second
    and tensor-core TFLOP/s."""
    import torch
    import llama_decode_forward_gb300 as L
    base = PREFILL_CFGS[args.prefill_weights]
    cfg = base.scaled(max_seq=PREFILL_N + 128)
    W = synth.make_weights(cfg)
    dec = L.Decoder(cfg, W)
    copy = args.prefill_f16_copy and args.prefill_weights == "q8_0"
    if copy:
        L.llm_prefill_f16_copy(dec.h)
    toks = synth.prompt(cfg, PREFILL_N)
    logits = np.empty(cfg.vocab, np.float32)
    for _ in range(max(args.warmup, 3)):
        L.llm_prefill(dec.h, toks, 0, logits)
    torch.cuda.synchronize()
    # CUDA events on the stream the library enqueues on (the handle's: the
    # legacy default stream), around each synchronous call
    st = torch.cuda.default_stream()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    t0 = time.perf_counter()
    for i in range(args.steps):
        starts[i].record(st)
        L.llm_prefill(dec.h, toks, 0, logits)
        ends[i].record(st)
    torch.cuda.synchronize()
    wall = time.perf_counter() - t0
    per = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    el = sum(per) / 1000.0
    fl = prefill_flops(cfg, PREFILL_N)
    tflops = fl * args.steps / el / 1e12
    peak = None
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            peak = json.load(f).get("bf16_tflops")
    what = {"f16": "Qwen2-style 1B-shape F16", "q8_0": "Llama-3.2-1B-shape Q8_0"}[args.prefill_weights]
    line = {"metric": f"prefill tok/s ({what}, 512 tokens from pos 0)",
            "value": PREFILL_N * args.steps / el, "unit": "tok/s", "n_gpus": 1, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": 1000.0 * el / args.steps, "higher_is_better": True,
            "dtype": "f16 operands, f32 accumulate",
            "data": f"synthetic (seeded random {args.prefill_weights.upper()} weights and tokens)",
            "config": {"workload": f"{base.name} prefill, 512 tokens", "flops_per_prefill": fl,
                       "q8_0_operands": ("F16 copy of the layer matrices (llm_prefill_f16_copy)" if copy
                                         else "expanded inside each GEMM") if args.prefill_weights == "q8_0" else None},
            "roofline": {"bound": "tensor", "achieved": tflops, "peak": peak, "unit": "TFLOP/s",
                         "frac": tflops / peak if peak else None,
                         "peak_source": "measured (MEASURED_PEAKS.json bf16_tflops; f16 taken equal)"},
            "launch_ms": percentiles(per),
            "timing": "CUDA events on the library's stream around each synchronous llm_prefill call (device time "
                      "from the token upload to the logits copy); host wall clock over the same calls: "
                      f"{1000.0 * wall / args.steps:.3f} ms per prefill"}
    dec.close()
    print(json.dumps(line))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--workload", choices=["decode", "prefill"], default="decode",
                    help="decode (the headline line) or the optional batched-prefill line")
    ap.add_argument("--prefill-weights", choices=sorted(PREFILL_CFGS), default="f16",
                    help="weight type of the prefill line's model")
    ap.add_argument("--prefill-f16-copy", action="store_true",
                    help="Q8_0 prefill line: give the handle its F16 copy of the layer matrices first")
    ap.add_argument("--model", choices=sorted(DECODE_MODELS), default="llama1b_q8",
                    help="decode workload's model: the Llama-3.2-1B shape (the headline) or the Llama-2-7B shape")
    ap.add_argument("--numerics", choices=["exact", "llamacpp"], default="exact",
                    help="the decode step's rounding (llm_config.numerics); llamacpp is not the headline")
    ap.add_argument("--pos", type=int, default=None,
                    help="position of the timed decode step (rows 0..pos-1 pre-filled); default 4095")
    args = ap.parse_args()
    if args.impl == "reference":
        return run_reference(args)
    if args.workload == "prefill":
        return run_prefill(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
