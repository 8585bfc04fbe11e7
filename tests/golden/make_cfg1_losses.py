"""Writes the oracle's loss trajectory for the GPT-2 124M fp32 workload.

Workload: GPT-2 124M (L=12, C=768, NH=12, V=50257 padded to Vp=50304, maxT=1024),
fp32, one fixed batch B=4, T=64 of uniform tokens, 10 AdamW steps overfitting it
(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, weight decay 0). Initial parameters:
the seeded init recipe of transformer_lm_gb300.inputs.gpt2_params. The step
(forward with mean cross-entropy, backward, AdamW) is the training loop of llm.c
"train_gpt2_fp32.cu" (gpt2_forward, gpt2_zero_grad, gpt2_backward, gpt2_update).

Calls only the oracle and the shared seeded input generators. Run from the repo
root:  python tests/golden/make_cfg1_losses.py
"""
import os
import sys

import numpy as np

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__)))))
import oracle  # noqa: E402
from transformer_lm_gb300 import inputs  # noqa: E402

SEED, B, T, STEPS = 101, 4, 64, 10
LR, B1, B2, EPS, WD = 1e-4, 0.9, 0.999, 1e-8, 0.0
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "cfg1_gpt2_124m_fp32_losses.txt")


def main():
    d = inputs.GPT2_124M
    params = inputs.gpt2_params(d, SEED).astype(np.float64)
    tok = inputs.tokens(SEED, 1, B, T, d.V)
    tgt = inputs.tokens(SEED, 2, B, T, d.V)
    model = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    m = np.zeros_like(params)
    v = np.zeros_like(params)
    losses = []
    for step in range(1, STEPS + 1):
        loss = model.forward(params, tok, tgt)
        grads = np.zeros_like(params)
        model.backward(grads)
        oracle.adamw(params, grads, m, v, LR, B1, B2, EPS, WD, step)
        losses.append(loss)
        print(step, repr(loss), flush=True)
    with open(OUT, "w") as f:
        f.write("# oracle loss trajectory, GPT-2 124M fp32, B=4 T=64, 10 AdamW steps on one batch\n")
        f.write(f"# seed={SEED} lr={LR} beta1={B1} beta2={B2} eps={EPS} wd={WD}\n")
        f.write("# written by tests/golden/make_cfg1_losses.py (oracle only)\n")
        for i, l in enumerate(losses):
            f.write(f"{i + 1} {l!r}\n")


if __name__ == "__main__":
    main()
