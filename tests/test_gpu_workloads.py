"""The step at the workloads' own sizes, through the C ABI.

  GPT-2 124M fp32, B=4, T=64, 10 AdamW steps on one batch: each step's loss
      against the oracle's trajectory in tests/golden (relative 1e-5, the fp32
      loss bound).
  GPT-2 124M bf16, B=8, T=1024 (the size bench.py times): the mean loss and
      every per-position loss, the gradient of each of the 16 parameter
      tensors (cosine >= 0.99, the bf16 bound) and the post-AdamW master
      weights against the oracle run at the same size on the host cores; the
      AdamW update on sampled parameters against the oracle's formula;
      gradient accumulation k=2 on one batch equal to k=1 bit for bit.
  GPT-2 350M bf16, B=1, T=1024 (the workload's T, reduced B) with gradient
      accumulation over 4 micro-steps: each micro-step's loss and the
      accumulated gradient against the oracle.

The oracle computes a B-sequence batch as B accumulation micro-steps of one
sequence each, seeded with dloss = 1/(B*T): the gradient of a mean over the
batch is the sum of the per-sequence gradients (the accumulation identity the
oracle's own tests pin), and the host memory stays that of one sequence.
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


def _oracle_batch_as_sequences(d, params, tok, tgt, k_outer=1):
    """Mean loss, per-position losses and the accumulated gradient of a (B, T)
    batch (dloss = 1/(k_outer*B*T)), one sequence at a time."""
    B, T = tok.shape
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, T)
    p64 = params.astype(np.float64)
    grads = np.zeros(params.size)
    losses = []
    for b in range(B):
        m.forward(p64, np.ascontiguousarray(tok[b:b + 1]), np.ascontiguousarray(tgt[b:b + 1]),
                  grad_accum_k=B * k_outer)
        losses.append(m.act("losses"))
        m.backward(grads)
    losses = np.concatenate(losses)
    return float(np.mean(losses)), losses, grads


def _cosine(a, b):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    na, nb = np.linalg.norm(a), np.linalg.norm(b)
    return 1.0 if na == 0 and nb == 0 else float(a @ b / (na * nb))


def _cosines(got, ref, d):
    a_all, b_all = _split(got, d), _split(ref, d)
    out = {}
    for name in inputs.PARAM_NAMES:
        a, b = a_all[name].astype(np.float64), b_all[name].astype(np.float64)
        na, nb = np.linalg.norm(a), np.linalg.norm(b)
        out[name] = 1.0 if na == 0 and nb == 0 else float(a @ b / (na * nb))
    return out


def test_124m_bf16_full_size_step():
    d = inputs.GPT2_124M
    B, T = 8, 1024
    lr, b1, b2, eps, wd = 6e-4, 0.9, 0.95, 1e-8, 0.1
    params = inputs.round_to_bf16(inputs.gpt2_params(d, 7))
    tok = inputs.tokens(7, 1, B, T, d.V)
    tgt = inputs.tokens(7, 2, B, T, d.V)
    G.gpt2_init(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1)
    G.gpt2_set_params(params)
    G.gpt2_zero_grad()
    loss = G.gpt2_forward(tok, tgt, B, T)
    losses = G.gpt2_get_losses(B * T)
    G.gpt2_backward()
    g = G.gpt2_get_grads()
    before = G.gpt2_get_master()
    G.gpt2_adamw(lr, b1, b2, eps, wd, 1)
    after = G.gpt2_get_master()
    # gradient accumulation on one batch, at this size (split-K reductions included)
    g1 = _grads_accumulated(tok, tgt, B, T, 1)
    g2 = _grads_accumulated(tok, tgt, B, T, 2)
    G.gpt2_free()
    _assert_accumulation_exact(g2, g1, d)

    # the oracle at the same size
    ref_loss, ref_losses, ref_g = _oracle_batch_as_sequences(d, params, tok, tgt)
    print(f"124M B=8 T=1024: loss {loss:.6f} oracle {ref_loss:.6f}; per-position max |diff| "
          f"{np.max(np.abs(losses - ref_losses)):.4f}")
    assert abs(loss - ref_loss) <= 2e-2
    assert abs(loss - np.log(d.V)) < 0.5  # near ln V at init
    assert np.max(np.abs(losses - ref_losses)) <= 0.1
    cos = _cosines(g, ref_g, d)
    print("124M B=8 T=1024 gradient cosine per tensor:", {k: round(v, 6) for k, v in cos.items()})
    for name, c in cos.items():
        assert c >= 0.99, (name, c)
    # post-AdamW master weights against the oracle's AdamW on the oracle's
    # gradient. The first AdamW step moves each weight by about lr * g/(|g|+eps):
    # where the exact gradient is zero (the key bias: softmax ignores a shift
    # common to all of a query's scores) or within the eps band, the oracle
    # moves it by ~0 and the bf16 path by +-lr on rounding noise, so those
    # elements (|g_ref| < 10 eps) are checked for their step size only.
    ref_p = params.astype(np.float64)
    mm, vv = np.zeros_like(ref_p), np.zeros_like(ref_p)
    oracle.adamw(ref_p, ref_g, mm, vv, lr, b1, b2, eps, wd, 1)
    band = np.abs(ref_g) < 10 * eps
    keep = ~band
    cos_p = {n: _cosine(_split(after, d)[n][k], _split(ref_p, d)[n][k])
             for n, k in zip(inputs.PARAM_NAMES, _split(keep, d).values())}
    step = (after - params).astype(np.float64) + lr * wd * params
    ref_step = (ref_p - params) + lr * wd * params
    cos_u = {n: _cosine(_split(step, d)[n][k], _split(ref_step, d)[n][k])
             for n, k in zip(inputs.PARAM_NAMES, _split(keep, d).values())}
    print(f"124M eps-band elements: {int(band.sum())} of {band.size}")
    print("124M post-AdamW master cosine per tensor:", {k: round(v, 6) for k, v in cos_p.items()})
    print("124M AdamW update cosine per tensor:", {k: round(v, 4) for k, v in cos_u.items()})
    for name, c in cos_p.items():
        assert c >= 0.99, (name, c)
    assert np.all(np.abs(step[band]) <= 1.01 * lr + 1e-7)
    # the update's sign agrees wherever the gradient carries weight: agreement
    # weighted by |g| (the step-1 update is lr * g/(|g|+eps) + decay)
    w = np.abs(ref_g)
    agree = float(np.sum(w * (np.sign(step) == np.sign(ref_step))) / np.sum(w))
    print(f"124M AdamW update sign agreement weighted by |g|: {agree:.5f}")
    assert agree >= 0.99
    # AdamW on sampled parameters: the oracle's update of the GPU's own gradients
    idx = np.random.default_rng(0).choice(g.size, 200000, replace=False)
    p = before[idx].astype(np.float64)
    mm, vv = np.zeros_like(p), np.zeros_like(p)
    oracle.adamw(p, g[idx].astype(np.float64), mm, vv, lr, b1, b2, eps, wd, 1)
    np.testing.assert_allclose(after[idx], p, rtol=1e-6, atol=1e-7)


def test_350m_bf16_grad_accumulation_4():
    """Four micro-steps of different batches accumulate (+=) the gradient of
    their sum: per-tensor cosine >= 0.99 against the oracle's accumulated
    gradient (the bf16 bound), at the workload's T = 1024 with B reduced to 1.
    On one repeated batch, k=4 equals k=1 up to the bf16 rounding of the three
    partial sums (x/4 + x/4 + x/4 is not exact)."""
    d = inputs.GPT2_350M
    B, T, K = 1, 1024, 4
    params = inputs.round_to_bf16(inputs.gpt2_params(d, 9))
    toks = [inputs.tokens(9, 2 * i + 1, B, T, d.V) for i in range(K)]
    tgts = [inputs.tokens(9, 2 * i + 2, B, T, d.V) for i in range(K)]
    G.gpt2_init(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1)
    G.gpt2_set_params(params)
    G.gpt2_zero_grad()
    G.gpt2_set_grad_accum(K)
    got_loss = []
    for tok, tgt in zip(toks, tgts):
        got_loss.append(G.gpt2_forward(tok, tgt, B, T))
        G.gpt2_backward()
    g = G.gpt2_get_grads()
    G.gpt2_set_grad_accum(1)
    # one batch repeated: k=4 against k=1
    g1 = _grads_accumulated(toks[0], tgts[0], B, T, 1)
    g4 = _grads_accumulated(toks[0], tgts[0], B, T, 4)
    G.gpt2_free()
    for name in inputs.PARAM_NAMES:
        a, b = _split(g4, d)[name], _split(g1, d)[name]
        if name == "wte":
            # two += per micro-step (classifier matmul, then the encoder
            # scatter) whose running sum is rounded to bf16 eight times: the
            # error scales with the parts, which may cancel, so it is bounded
            # by the tensor's scale (eight roundings of up to 2^-9 each)
            ratio = float(np.max(np.abs(a - b)) / np.max(np.abs(b)))
            print(f"350M wte k=4 vs k=1: max |diff| / max |g| = {ratio:.2e}, cosine {_cosine(a, b):.7f}")
            assert ratio <= 8 * 2.0 ** -9, name
            assert _cosine(a, b) > 0.9999, name
        else:
            assert np.all(np.abs(a - b) <= 2.0 ** -7 * np.abs(b) + 2.0 ** -7 * 1e-3 * np.max(np.abs(b))), name
    # oracle: the four micro-batches, each seeded with dloss = 1/(K*B*T)
    ref = np.zeros(params.size)
    for i, (tok, tgt) in enumerate(zip(toks, tgts)):
        ref_loss, _, gi = _oracle_batch_as_sequences(d, params, tok, tgt, k_outer=K)
        ref += gi
        assert abs(got_loss[i] - ref_loss) <= 2e-2, (i, got_loss[i], ref_loss)
    cos = _cosines(g, ref, d)
    print("350M B=1 T=1024 k=4 gradient cosine per tensor:", {k: round(v, 6) for k, v in cos.items()})
    for name, c in cos.items():
        assert c >= 0.99, (name, c)


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
