"""Benchmark: one GPT-2 training step (forward, backward, AdamW) per iteration.

Workload: GPT-2 124M (L=12, C=768, NH=12, V=50257 padded to Vp=50304),
bf16 mixed precision (bf16 activations/params/grads, fp32 master weights and
AdamW moments), B=8, T=1024, AdamW lr 6e-4, wd 0.1, synthetic uniform tokens.

Prints ONE JSON line on rank 0. `value` is tokens/s with the token batch
already resident in HBM; `e2e` is the same metric through the host-pointer
C-ABI call (token upload and the loss read-back inside the timed region).
With --gpus N (under torchrun) every rank trains its own replica (the step has
no exchange on one GPU per replica); value = all ranks' tokens / max time.

--impl reference times the CPU oracle (the reference arm of this build) on a
bounded sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "GPT-2 train-step tokens/sec on 1 GB300; % of tensor/HBM roofline"
WORKLOAD = ("GPT-2 124M (L=12 C=768 NH=12 V=50257 Vp=50304) bf16 mixed-precision train step "
            "(fwd+bwd+AdamW lr 6e-4 wd 0.1), B=8 T=1024")
L, C, NH, V, Vp, MAXT = 12, 768, 12, 50257, 50304, 1024
B, T = 8, 1024
ACCUM = 1  # gradient-accumulation micro-steps per AdamW update
DIMS = "GPT2_124M"
LR, B1, B2, EPS, WD = 6e-4, 0.9, 0.95, 1e-8, 0.1


def select_model(name: str) -> None:
    """--model 350m: GPT-2 350M, B=16, T=1024, 4 micro-steps per update."""
    global L, C, NH, B, ACCUM, DIMS, WORKLOAD
    if name == "350m":
        L, C, NH, B, ACCUM, DIMS = 24, 1024, 16, 16, 4, "GPT2_350M"
        WORKLOAD = ("GPT-2 350M (L=24 C=1024 NH=16 V=50257 Vp=50304) bf16 mixed-precision train step "
                    "(4 micro-steps of B=16 T=1024 with += gradient accumulation, then AdamW lr 6e-4 "
                    "wd 0.1)")


def model_flops_per_token() -> float:
    """6 * (matmul weights, unpadded vocab) + causal attention fwd+bwd: 6 L C T."""
    n_mm = 12 * L * C * C + C * V
    return 6.0 * n_mm + 6.0 * L * C * T


def gemm_traffic():
    """DRAM bytes per GEMM launch from the committed ncu summary, or None when
    the GEMM source has changed since those counters were taken."""
    import hashlib
    root = os.path.dirname(os.path.abspath(__file__))
    try:
        text = open(os.path.join(root, "profiles", "roofline_gemm_step.md")).read()
        src = open(os.path.join(root, "transformer_lm_gb300", "csrc", "gemm_tc.cu"), "rb").read()
    except OSError:
        return None
    vals = dict(line.split(":", 1) for line in text.splitlines()
                if line.startswith(("traffic_bytes_per_launch:", "source_sha256_16:")))
    if vals.get("source_sha256_16", "").strip() != hashlib.sha256(src).hexdigest()[:16]:
        return None
    return float(vals["traffic_bytes_per_launch"])


def load_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", d["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"bench_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200"], stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
        try:
            os.remove(self.path)
        except OSError:
            pass
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def dist_setup(backend: str | None = None):
    """One process per GPU (torchrun's RANK / LOCAL_RANK / WORLD_SIZE). The
    replicas exchange nothing on the data path: the process group only carries
    the barriers and the max-over-ranks of the timings (NCCL on GPUs, gloo
    when there is no GPU)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch
        import torch.distributed as dist
        if backend is None:
            backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(tokens_per_rank: int, world: int, seconds: float) -> float:
    """Whole-job tokens/s: every rank's tokens over the slowest rank's time."""
    return world * tokens_per_rank / seconds


# --------------------------------------------------------------------------- CPU oracle arm
ORACLE_SAMPLE_T = 256


def oracle_sample_setup(seed: int = 1337):
    """The oracle on a bounded sample of the workload: the full 124M model and
    AdamW over all its parameters, on a batch of B=1, T=ORACLE_SAMPLE_T tokens."""
    import numpy as np

    import oracle
    from transformer_lm_gb300 import inputs
    d = getattr(inputs, DIMS)
    params = inputs.round_to_bf16(inputs.gpt2_params(d, seed)).astype(np.float64)
    tok = inputs.tokens(42, 1, 1, ORACLE_SAMPLE_T, d.V)
    tgt = inputs.tokens(42, 2, 1, ORACLE_SAMPLE_T, d.V)
    model = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, ORACLE_SAMPLE_T)
    state = dict(params=params, grads=np.zeros_like(params), m=np.zeros_like(params),
                 v=np.zeros_like(params), tok=tok, tgt=tgt, model=model, step=0)
    return state


def oracle_sample_step(st) -> None:
    import oracle
    st["grads"][:] = 0.0
    st["model"].forward(st["params"], st["tok"], st["tgt"])
    st["model"].backward(st["grads"])
    st["step"] += 1
    oracle.adamw(st["params"], st["grads"], st["m"], st["v"], LR, B1, B2, EPS, WD, st["step"])


def cpu_baseline(steps: int = 1) -> dict:
    import oracle
    st = oracle_sample_setup()
    t0 = time.perf_counter()
    for _ in range(steps):
        oracle_sample_step(st)
    dt = time.perf_counter() - t0
    return {"value": steps * ORACLE_SAMPLE_T / dt, "unit": "tokens/s", "cores": oracle.num_threads(),
            "kind": "oracle",
            "sample": (f"full {DIMS[5:]} model fwd+bwd on B=1 T={ORACLE_SAMPLE_T} plus AdamW over "
                       f"all params, {steps} step(s), fp64, {dt:.1f} s")}


def run_reference(args):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    import oracle
    st = oracle_sample_setup()
    for _ in range(args.warmup):
        oracle_sample_step(st)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_sample_step(st)
    dt = time.perf_counter() - t0
    value = args.steps * ORACLE_SAMPLE_T / dt
    sample = (f"each step: full {DIMS[5:]} model fwd+bwd on B=1 T={ORACLE_SAMPLE_T} plus AdamW over "
              f"all params, fp64 CPU oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * dt / args.steps, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD + f" (sampled: B=1 T={ORACLE_SAMPLE_T} per step)",
                       "global_batch": 1, "seq_len": ORACLE_SAMPLE_T, "parallelism": "none"},
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": oracle.num_threads(),
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# --------------------------------------------------------------------------- GPU arm
def run_ours(args):
    world, rank, local = dist_setup()
    import numpy as np
    import torch

    from transformer_lm_gb300 import gpt2 as G
    from transformer_lm_gb300 import inputs

    torch.cuda.set_device(local)
    peaks = load_peaks()
    # baseline first, on rank 0 only, at N=1 only, before any GPU work
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(2)

    G.gpt2_init(L, C, NH, V, Vp, MAXT, 1337 + rank)
    # a created stream (the legacy default stream has handle 0, which the
    # library reads as "use your own stream"); torch events are recorded on it
    stream = torch.cuda.Stream()
    torch.cuda.set_stream(stream)
    G.gpt2_set_stream(stream.cuda_stream)
    G.gpt2_set_grad_accum(ACCUM)
    # ACCUM micro-batches of B x T ids, one after another
    tok = inputs.tokens(42 + rank, 1, ACCUM * B, T, V)
    tgt = inputs.tokens(42 + rank, 2, ACCUM * B, T, V)
    d_tok = torch.from_numpy(tok.reshape(-1)).cuda()
    d_tgt = torch.from_numpy(tgt.reshape(-1)).cuda()
    d_loss = torch.zeros(ACCUM, device="cuda")
    step_no = [0]

    # pinned host copies of the batch for the end-to-end leg
    h_tok = torch.from_numpy(tok.reshape(-1)).pin_memory()
    h_tgt = torch.from_numpy(tgt.reshape(-1)).pin_memory()

    def device_step():
        # forward + zero_grad + backward + AdamW; replayed from a CUDA graph
        # once the first call has recorded it
        step_no[0] += 1
        G.gpt2_train_step(d_tok, d_tgt, B, T, LR, B1, B2, EPS, WD, step_no[0], d_loss)

    def host_step():
        # the batch goes up from pinned host memory and the loss comes back
        d_tok.copy_(h_tok, non_blocking=True)
        d_tgt.copy_(h_tgt, non_blocking=True)
        device_step()
        return float(d_loss.cpu().mean())

    for _ in range(args.warmup):
        device_step()
    G.gpt2_sync()

    # ---- device-resident timed region
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    launches0 = G.gpt2_launch_count()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        device_step()
    ev1.record(stream)
    torch.cuda.synchronize()
    launches = G.gpt2_launch_count() - launches0
    clk = clocks.stop()
    barrier(world)
    ms = ev0.elapsed_time(ev1)
    ms = max_over_ranks(ms, world)
    G.gpt2_sync()
    loss_dev = float(d_loss.cpu().mean())

    # ---- per-kernel durations: CUDA events around every launch, on the
    # library's stream, over a second pass of the same steps (kept out of
    # the timed region above because the extra event records slow the step)
    G.gpt2_timing_begin(args.steps * 500 * ACCUM * L // 12)
    for _ in range(args.steps):
        device_step()
    G.gpt2_timing_end()

    # ---- end-to-end: host tokens in, loss read back, every step
    for _ in range(2):
        host_step()
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        loss_host = host_step()
    torch.cuda.synchronize()
    e2e_s = max_over_ranks(time.perf_counter() - t0, world)
    G.gpt2_sync()

    tokens_all = world * ACCUM * B * T * args.steps
    value = job_throughput(ACCUM * B * T * args.steps, world, ms / 1000.0)
    e2e_value = job_throughput(ACCUM * B * T * args.steps, world, e2e_s)
    step_flops = model_flops_per_token() * ACCUM * B * T

    fam = {}
    for f in G.FAMILIES:
        t_ms, n, work = G.gpt2_timing_get(f)
        fam[f] = dict(ms=t_ms, launches=n, work=work)
    g = fam["gemm"]
    gemm_tflops = g["work"] / (g["ms"] / 1000.0) / 1e12 if g["ms"] > 0 else None
    peak_t = peaks["bf16_tflops_sustained"]
    roofline = {"bound": "tensor", "kernel": "gemm_tc_k (tcgen05 bf16 GEMM, all launches)",
                "achieved": gemm_tflops, "peak": peak_t, "unit": "TFLOP/s",
                "frac": (gemm_tflops / peak_t) if gemm_tflops else None,
                "peak_source": f"{peaks['source']} bf16_tflops_sustained",
                "traffic": gemm_traffic(),
                "per_launch_gflop": g["work"] / max(g["launches"], 1) / 1e9,
                "avg_launch_ms": g["ms"] / max(g["launches"], 1)}
    breakdown = {f: {"ms_per_step": v["ms"] / args.steps, "launches_per_step": v["launches"] / args.steps}
                 for f, v in fam.items() if v["launches"]}
    for f in ("ln_fwd", "ln_bwd", "classifier", "adamw", "encoder"):
        if fam[f]["ms"] > 0:
            breakdown[f]["gb_per_s"] = fam[f]["work"] / (fam[f]["ms"] / 1000.0) / 1e9
    for f in ("attn_fwd", "attn_bwd"):
        if fam[f]["ms"] > 0:
            breakdown[f]["tflop_per_s"] = fam[f]["work"] / (fam[f]["ms"] / 1000.0) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "global_batch": ACCUM * B * world, "seq_len": T,
                   "parallelism": "replicas" if world > 1 else "single",
                   "l2": "no flush: per-step working set (~6 GB) is larger than L2"},
        "mfu": step_flops / (ms / 1000.0 / args.steps) / (peaks["bf16_tflops_sustained"] * 1e12),
        "mfu_vs_burst_peak": step_flops / (ms / 1000.0 / args.steps) / (peaks["bf16_tflops"] * 1e12),
        "model_tflop_per_step": step_flops / 1e12,
        "roofline": roofline,
        "breakdown": breakdown,
        "e2e": {"value": e2e_value, "unit": "tokens/s", "h2d_bytes_per_step": 2 * ACCUM * B * T * 4,
                "d2h_bytes_per_step": 4 * ACCUM},
        "gpu_launches": launches,
        "clocks": clk,
        "loss": {"device_path": loss_dev, "host_path": loss_host},
    }
    if cpu is not None:
        line["cpu_baseline"] = cpu
    if rank == 0:
        print(json.dumps(line), flush=True)
    G.gpt2_free()
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--model", default="124m", choices=["124m", "350m"],
                    help="124m: the headline workload (B=8, T=1024); 350m: B=16, T=1024, "
                         "4 accumulation micro-steps per update")
    args = ap.parse_args()
    select_model(args.model)
    if args.warmup < 3 and args.impl == "ours":
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
