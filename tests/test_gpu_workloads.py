"""The step at the workloads' own sizes, through the C ABI.

  GPT-2 124M fp32, B=4, T=64, 10 AdamW steps on one batch: each step's loss
      against the oracle's trajectory in tests/golden (relative 1e-5, the fp32
      loss bound).
  GPT-2 124M bf16, B=8, T=1024 (the size bench.py times): per-position losses
      of one sequence prefix against the oracle (a causal model's loss at
      position t depends only on tokens 0..t, so the oracle runs the prefix
      alone); the AdamW update on sampled parameters against the oracle's
      formula; gradient accumulation k=2 on one batch equal to k=1 bit for bit.
  GPT-2 350M bf16 with gradient accumulation over 4 micro-steps: each
      micro-step's loss and the accumulated gradient against the oracle.
"""
import os

import numpy as np
import pytest

import oracle
from transformer_lm_gb300 import inputs
from transformer_lm_gb300 import gpt2 as G

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                      "cfg1_gpt2_124m_fp32_losses.txt")


def _golden_losses():
    vals = []
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        vals.append(float(line.split()[1]))
    return np.array(vals)


def test_124m_fp32_loss_trajectory_matches_oracle():
    """The trajectory written by tests/golden/make_cfg1_losses.py (same seed,
    batch and AdamW settings)."""
    ref = _golden_losses()
    d = inputs.GPT2_124M
    B, T = 4, 64
    params = inputs.gpt2_params(d, 101)
    tok = inputs.tokens(101, 1, B, T, d.V)
    tgt = inputs.tokens(101, 2, B, T, d.V)
    G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, G.GPT2_FP32, 0)
    G.gpt2_set_params(params)
    got = []
    for step in range(1, len(ref) + 1):
        got.append(G.gpt2_forward(tok, tgt, B, T))
        G.gpt2_zero_grad()
        G.gpt2_backward()
        G.gpt2_adamw(1e-4, 0.9, 0.999, 1e-8, 0.0, step)
    G.gpt2_sync()
    G.gpt2_free()
    got = np.array(got)
    assert ref[-1] < ref[0]  # the batch is being fitted
    np.testing.assert_allclose(got, ref, rtol=1e-5, atol=0)


def _prefix_losses(d, params, tok, tgt, t_prefix):
    """Oracle per-position losses of sequence 0's first t_prefix positions."""
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, t_prefix)
    m.forward(params.astype(np.float64), np.ascontiguousarray(tok[:1, :t_prefix]),
              np.ascontiguousarray(tgt[:1, :t_prefix]))
    return m.act("losses").reshape(-1)


def _split(flat, d):
    out, off = {}, 0
    for name, s in zip(inputs.PARAM_NAMES, inputs.param_sizes(d)):
        out[name] = flat[off:off + s]
        off += s
    return out


def _grads_accumulated(tok, tgt, B, T, k):
    G.gpt2_zero_grad()
    G.gpt2_set_grad_accum(k)
    for _ in range(k):
        G.gpt2_forward(tok, tgt, B, T)
        G.gpt2_backward()
    G.gpt2_set_grad_accum(1)
    return G.gpt2_get_grads()


def _assert_accumulation_exact(g_k, g_1, d):
    """k micro-steps on one batch, each seeded with dloss/k, equal one step:
    scaling by a power of two is exact and a value rounded once absorbs its own
    fractions, for every tensor that takes one += per backward. wte takes two
    (classifier matmul, then the encoder scatter) and is double-rounded."""
    a_all, b_all = _split(g_k, d), _split(g_1, d)
    for name in inputs.PARAM_NAMES:
        a, b = a_all[name], b_all[name]
        if name == "wte":
            assert np.max(np.abs(a - b)) <= 2.0 ** -7 * np.max(np.abs(b)), name
        else:
            assert np.array_equal(a, b), name


def test_124m_bf16_full_size_step():
    d = inputs.GPT2_124M
    B, T = 8, 1024
    params = inputs.round_to_bf16(inputs.gpt2_params(d, 7))
    tok = inputs.tokens(7, 1, B, T, d.V)
    tgt = inputs.tokens(7, 2, B, T, d.V)
    G.gpt2_init(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1)
    G.gpt2_set_params(params)
    # per-position losses of a 256-token prefix against the oracle
    G.gpt2_zero_grad()
    loss = G.gpt2_forward(tok, tgt, B, T)
    got = G.gpt2_get_losses(B * T).reshape(B, T)[0, :256]
    ref = _prefix_losses(d, params, tok, tgt, 256)
    assert abs(float(np.mean(got)) - float(np.mean(ref))) <= 2e-2
    assert np.max(np.abs(got - ref)) <= 0.1
    assert abs(loss - np.log(d.V)) < 0.5  # near ln V at init
    # AdamW on sampled parameters: the oracle's update of the master weights
    G.gpt2_backward()
    g = G.gpt2_get_grads()
    before = G.gpt2_get_master()
    G.gpt2_adamw(6e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    after = G.gpt2_get_master()
    idx = np.random.default_rng(0).choice(g.size, 200000, replace=False)
    p = before[idx].astype(np.float64)
    mm, vv = np.zeros_like(p), np.zeros_like(p)
    oracle.adamw(p, g[idx].astype(np.float64), mm, vv, 6e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    np.testing.assert_allclose(after[idx], p, rtol=1e-6, atol=1e-7)
    # gradient accumulation on one batch, at this size (split-K reductions included)
    g1 = _grads_accumulated(tok, tgt, B, T, 1)
    g2 = _grads_accumulated(tok, tgt, B, T, 2)
    _assert_accumulation_exact(g2, g1, d)
    G.gpt2_free()


def test_350m_bf16_grad_accumulation_4():
    """Four micro-steps of different batches accumulate (+=) the gradient of
    their sum: per-tensor cosine >= 0.99 against the oracle's accumulated
    gradient (the bf16 bound). On one repeated batch, k=4 equals k=1 up to the
    bf16 rounding of the three partial sums (x/4 + x/4 + x/4 is not exact)."""
    d = inputs.GPT2_350M
    B, T, K = 1, 64, 4
    params = inputs.round_to_bf16(inputs.gpt2_params(d, 9))
    toks = [inputs.tokens(9, 2 * i + 1, B, T, d.V) for i in range(K)]
    tgts = [inputs.tokens(9, 2 * i + 2, B, T, d.V) for i in range(K)]
    # oracle: the four micro-batches, each seeded with dloss = 1/(K*B*T)
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    ref = np.zeros(params.size)
    ref_loss = []
    for tok, tgt in zip(toks, tgts):
        ref_loss.append(m.forward(params.astype(np.float64), tok, tgt, grad_accum_k=K))
        m.backward(ref)
    G.gpt2_init(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1)
    G.gpt2_set_params(params)
    G.gpt2_zero_grad()
    G.gpt2_set_grad_accum(K)
    for i, (tok, tgt) in enumerate(zip(toks, tgts)):
        loss = G.gpt2_forward(tok, tgt, B, T)
        assert abs(loss - ref_loss[i]) <= 2e-2, (i, loss, ref_loss[i])
        G.gpt2_backward()
    g = G.gpt2_get_grads()
    G.gpt2_set_grad_accum(1)
    got, want = _split(g, d), _split(ref, d)
    for name in inputs.PARAM_NAMES:
        a, b = got[name].astype(np.float64), want[name]
        c = float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b) + 1e-300))
        assert c >= 0.99, (name, c)
    # one batch repeated: k=4 against k=1
    g1 = _grads_accumulated(toks[0], tgts[0], B, T, 1)
    g4 = _grads_accumulated(toks[0], tgts[0], B, T, 4)
    for name in inputs.PARAM_NAMES:
        a, b = _split(g4, d)[name], _split(g1, d)[name]
        assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 2.0 ** -7 * 1e-3 * np.max(np.abs(b))), name
    G.gpt2_free()


def test_fused_op_full_size_sampled_rows():
    """x [1024, 8192], W [8192, 8192], b [8192]: each output row depends on its
    x row and all of W, so the oracle computes a sample of rows alone; every
    element within 1e-3 relative."""
    import torch
    M, K, N = 1024, 8192, 8192
    x, W, b = inputs.fused_op_inputs(M, K, N, seed=5)
    out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    G.fused_linear_bias_gelu_softmax(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(),
                                     torch.from_numpy(b).cuda(), out, M, K, N)
    G.gpt2_device_status()
    y = out.cpu().numpy()
    np.testing.assert_allclose(y.sum(1), 1.0, atol=1e-4)
    rows = np.array([0, 1, 511, 777, 1023])
    ref = oracle.fused_linear_bias_gelu_softmax(np.ascontiguousarray(x[rows]), W, b)
    rel = np.max(np.abs(y[rows] - ref) / np.abs(ref))
    print("fused op, sampled rows: max elementwise relative error", rel)
    assert rel < 1e-3
