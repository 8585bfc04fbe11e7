"""Time one kernel of libgpt2.so on synthetic inputs (for profiling and tuning).

    python -m transformer_lm_gb300.kernel_bench gemm M N K [a_kmajor b_kmajor epilogue] [--reps R]
    python -m transformer_lm_gb300.kernel_bench attention B T C NH [--reps R]
    python -m transformer_lm_gb300.kernel_bench fused M K N [--reps R]
    python -m transformer_lm_gb300.kernel_bench layernorm N C [--reps R]

Prints the mean CUDA-event time per launch and the throughput. Inputs are
allocated with torch; the kernels run through the C ABI on torch's current
stream. --graph captures the R calls in a CUDA graph and times its replays,
which leaves out the host's per-call cost.
"""
from __future__ import annotations

import argparse
import sys


_GRAPH = False


def _time(fn, reps):
    import torch
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            fn()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    if _GRAPH:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(reps):
                fn()
        with torch.cuda.stream(s):
            g.replay()
            e0.record()
            for _ in range(3):
                g.replay()
            e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / (3 * reps)
    with torch.cuda.stream(s):
        e0.record()
        for _ in range(reps):
            fn()
        e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


def _cur():
    import torch
    return torch.cuda.current_stream().cuda_stream


def main(argv=None):
    import torch

    from transformer_lm_gb300 import gpt2 as G
    ap = argparse.ArgumentParser()
    ap.add_argument("kind", choices=["gemm", "attention", "fused", "layernorm"])
    ap.add_argument("dims", nargs="*")
    ap.add_argument("--reps", type=int, default=20)
    ap.add_argument("--graph", action="store_true")
    a = ap.parse_args(argv)
    global _GRAPH
    _GRAPH = a.graph
    d = a.dims
    if a.kind == "gemm":
        M, N, K = int(d[0]), int(d[1]), int(d[2])
        akm = int(d[3]) if len(d) > 3 else 1
        bkm = int(d[4]) if len(d) > 4 else 1
        epi = d[5] if len(d) > 5 else "store"
        A = (torch.randn(M * K, device="cuda") * 0.5).bfloat16()
        B = (torch.randn(N * K, device="cuda") * 0.05).bfloat16()
        D = torch.zeros(M * N, device="cuda").bfloat16()
        D2 = torch.zeros(M * N, device="cuda").bfloat16() if epi == "gelu" else None
        aux = torch.randn(M * N, device="cuda").bfloat16() if epi in ("resid", "gelu_bwd") else None
        bias = torch.zeros(N, device="cuda").bfloat16()
        ws = torch.empty(16 * M * N, device="cuda")  # split-K scratch for "accum"

        def fn():
            G.gpt2_gemm(G.GPT2_BF16, 1, epi, A, K if akm else M, akm, B, K if bkm else N, bkm, D, N,
                        bias=bias, aux=aux, ldaux=N, D2=D2, M=M, N=N, K=K, ws=ws,
                        ws_floats=ws.numel(), stream=_cur())
        ms = _time(fn, a.reps)
        print(f"gemm {M}x{N}x{K} a_kmajor={akm} b_kmajor={bkm} {epi}: {ms * 1e3:.1f} us, "
              f"{2.0 * M * N * K / ms / 1e9:.1f} TFLOP/s")
    elif a.kind == "attention":
        B, T, C, NH = (int(x) for x in d[:4])
        qkv = (torch.randn(B * T * 3 * C, device="cuda")).bfloat16()
        out = torch.zeros(B * T * C, device="cuda").bfloat16()
        lse = torch.zeros(B * NH * T, device="cuda")
        dout = (torch.randn(B * T * C, device="cuda") * 0.1).bfloat16()
        dqkv = torch.zeros(B * T * 3 * C, device="cuda").bfloat16()
        Dsc = torch.zeros(B * NH * T, device="cuda")
        flops = 2.0 * B * NH * T * (T + 1) * (C // NH)
        ms_f = _time(lambda: G.gpt2_attention_forward(1, 1, qkv, out, lse, B, T, C, NH, _cur()),
                     a.reps)
        ms_b = _time(lambda: G.gpt2_attention_backward(1, 1, dout, qkv, out, lse, dqkv, Dsc, B, T, C,
                                                       NH, _cur()), a.reps)
        print(f"attention B={B} T={T} C={C} NH={NH}: fwd {ms_f * 1e3:.1f} us "
              f"({flops / ms_f / 1e9:.1f} TFLOP/s), bwd {ms_b * 1e3:.1f} us "
              f"({2 * flops / ms_b / 1e9:.1f} TFLOP/s)")
    elif a.kind == "layernorm":
        N, C = int(d[0]), int(d[1])
        x = torch.randn(N * C, device="cuda").bfloat16()
        w = torch.ones(C, device="cuda").bfloat16()
        b = torch.zeros(C, device="cuda").bfloat16()
        y = torch.empty_like(x)
        mean = torch.empty(N, device="cuda")
        rstd = torch.empty(N, device="cuda")
        dy = (torch.randn(N * C, device="cuda") * 0.01).bfloat16()
        dx = torch.zeros_like(x)
        dw = torch.zeros_like(w)
        db = torch.zeros_like(b)
        scratch = torch.zeros(G.gpt2_layernorm_backward_scratch_floats(C), device="cuda")
        ms_f = _time(lambda: G.gpt2_layernorm_forward(1, y, mean, rstd, x, w, b, N, C, _cur()), a.reps)
        ms_b = _time(lambda: G.gpt2_layernorm_backward(1, dx, dw, db, dy, x, w, mean, rstd, N, C, 1,
                                                       scratch, _cur()), a.reps)
        print(f"layernorm N={N} C={C}: fwd {ms_f * 1e3:.1f} us ({4.0 * N * C / ms_f / 1e6:.0f} GB/s), "
              f"bwd {ms_b * 1e3:.1f} us ({8.0 * N * C / ms_b / 1e6:.0f} GB/s)")
    else:
        M, K, N = int(d[0]), int(d[1]), int(d[2])
        x = torch.randn(M, K, device="cuda")
        W = torch.randn(N, K, device="cuda") / K ** 0.5
        b = (torch.rand(N, device="cuda") - 0.5) * 0.2
        y = torch.empty(M, N, device="cuda")
        ms = _time(lambda: G.fused_linear_bias_gelu_softmax(x, W, b, y, M, K, N, _cur()), a.reps)
        print(f"fused {M}x{K}x{N}: {ms * 1e3:.1f} us, {2.0 * M * N * K / ms / 1e9:.1f} TFLOP/s")
    G.gpt2_device_status()
    return 0


if __name__ == "__main__":
    sys.exit(main())
