"""Pins for the CPU oracle: each test ties one oracle function to something
other than itself -- a library routine (torch float64), a closed form, a
finite-difference derivative, or an invariant the method guarantees."""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from transformer_lm_gb300 import inputs

TINY = inputs.TINY


def _tiny_model(B=2, T=32, d=TINY):
    return oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)


# --------------------------------------------------------------------------
# parameter layout


def test_param_count_matches_published_gpt2_sizes():
    # GPT-2 small has 124,439,808 parameters with the 50257-token vocabulary;
    # padding wte to 50304 rows adds 47*768.
    _, total = oracle.param_sizes(12, 768, 12, 50257, 50257, 1024)
    assert total == 124_439_808
    _, total = oracle.param_sizes(12, 768, 12, 50257, 50304, 1024)
    assert total == 124_475_904
    # GPT-2 medium: 354,823,168 with the unpadded vocabulary
    _, total = oracle.param_sizes(24, 1024, 16, 50257, 50257, 1024)
    assert total == 354_823_168


def test_param_sizes_agree_with_input_generator():
    for d in (inputs.TINY, inputs.GPT2_124M, inputs.GPT2_350M):
        sizes, total = oracle.param_sizes(d.L, d.C, d.NH, d.V, d.Vp, d.maxT)
        assert sizes == inputs.param_sizes(d)


# --------------------------------------------------------------------------
# single operations against torch float64


def test_layernorm_forward_matches_torch_and_normalises():
    rng = np.random.default_rng(0)
    x = rng.normal(size=(37, 64)) * 3 + 1.5
    w = rng.normal(size=64)
    b = rng.normal(size=64)
    y, mean, rstd = oracle.layernorm_forward(x, w, b)
    ref = F.layer_norm(torch.tensor(x), (64,), torch.tensor(w), torch.tensor(b), eps=1e-5)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-12)
    # pre-affine output: zero mean, variance 1 - O(eps/var)
    yn, _, _ = oracle.layernorm_forward(x, np.ones(64), np.zeros(64))
    assert np.abs(yn.mean(axis=1)).max() < 1e-12
    var = x.var(axis=1)
    np.testing.assert_allclose(yn.var(axis=1), var / (var + 1e-5), rtol=1e-12)
    np.testing.assert_allclose(mean, x.mean(axis=1), rtol=1e-12)


def test_layernorm_backward_matches_autograd_and_accumulates():
    rng = np.random.default_rng(1)
    N, C = 19, 48
    x = rng.normal(size=(N, C))
    w = rng.normal(size=C)
    b = rng.normal(size=C)
    dy = rng.normal(size=(N, C))
    _, mean, rstd = oracle.layernorm_forward(x, w, b)
    dinp0 = rng.normal(size=(N, C))
    dw0 = rng.normal(size=C)
    db0 = rng.normal(size=C)
    dinp, dw, db = dinp0.copy(), dw0.copy(), db0.copy()
    oracle.layernorm_backward(dinp, dw, db, dy, x, w, mean, rstd)
    xt = torch.tensor(x, requires_grad=True)
    wt = torch.tensor(w, requires_grad=True)
    bt = torch.tensor(b, requires_grad=True)
    F.layer_norm(xt, (C,), wt, bt, eps=1e-5).backward(torch.tensor(dy))
    np.testing.assert_allclose(dinp - dinp0, xt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dw - dw0, wt.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(db - db0, bt.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_gelu_tanh_against_torch_and_exact_gelu():
    x = np.linspace(-8, 8, 2001)
    y = oracle.gelu_forward(x)
    ref = F.gelu(torch.tensor(x), approximate="tanh").numpy()
    np.testing.assert_allclose(y, ref, rtol=1e-14, atol=1e-15)
    # odd-part identity of the tanh form: gelu(x) - gelu(-x) = x
    np.testing.assert_allclose(y - oracle.gelu_forward(-x), x, rtol=0, atol=1e-14)
    assert oracle.gelu_forward(np.zeros(1))[0] == 0.0
    # it approximates x * Phi(x) to well within 1e-3
    from scipy.special import ndtr
    assert np.abs(y - x * ndtr(x)).max() < 1e-3


def test_gelu_backward_matches_autograd_and_finite_differences():
    x = np.linspace(-6, 6, 1201)
    dout = np.cos(x)
    d = oracle.gelu_backward(x, dout)
    xt = torch.tensor(x, requires_grad=True)
    F.gelu(xt, approximate="tanh").backward(torch.tensor(dout))
    np.testing.assert_allclose(d, xt.grad.numpy(), rtol=1e-12, atol=1e-14)
    h = 1e-6
    fd = (oracle.gelu_forward(x + h) - oracle.gelu_forward(x - h)) / (2 * h) * dout
    np.testing.assert_allclose(d, fd, rtol=1e-6, atol=1e-8)


def test_matmul_forward_backward_against_numpy():
    rng = np.random.default_rng(2)
    N, Cin, Cout = 13, 21, 17
    x = rng.normal(size=(N, Cin))
    w = rng.normal(size=(Cout, Cin))
    bias = rng.normal(size=Cout)
    y = oracle.matmul_forward(x, w, bias)
    np.testing.assert_allclose(y, x @ w.T + bias, rtol=1e-12, atol=1e-12)
    dy = rng.normal(size=(N, Cout))
    dw = np.ones((Cout, Cin))
    db = np.ones(Cout)
    dx = oracle.matmul_backward(dy, x, w, dw, db)
    np.testing.assert_allclose(dx, dy @ w, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(dw, 1.0 + dy.T @ x, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(db, 1.0 + dy.sum(0), rtol=1e-12, atol=1e-12)


def _qkv_to_torch(qkv, B, T, C, NH):
    HS = C // NH
    t = torch.tensor(qkv).view(B, T, 3, NH, HS)
    return t[:, :, 0].transpose(1, 2), t[:, :, 1].transpose(1, 2), t[:, :, 2].transpose(1, 2)


@pytest.mark.parametrize("B,T,C,NH", [(2, 17, 32, 4), (1, 1, 16, 2), (3, 40, 64, 4)])
def test_attention_forward_matches_sdpa(B, T, C, NH):
    rng = np.random.default_rng(3)
    qkv = rng.normal(size=(B * T * 3 * C,))
    out, att = oracle.attention_forward(qkv, B, T, C, NH)
    q, k, v = _qkv_to_torch(qkv, B, T, C, NH)
    ref = F.scaled_dot_product_attention(q, k, v, is_causal=True)
    ref = ref.transpose(1, 2).reshape(-1).numpy()
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)
    A = att.reshape(B, NH, T, T)
    np.testing.assert_allclose(A.sum(-1), 1.0, rtol=0, atol=1e-12)
    assert np.all(np.triu(np.ones((T, T)), 1)[None, None] * A == 0.0)
    if T == 1:
        # one position: the output is v itself
        np.testing.assert_array_equal(out, v.transpose(1, 2).reshape(-1).numpy())


def test_attention_backward_matches_autograd():
    B, T, C, NH = 2, 23, 32, 4
    rng = np.random.default_rng(4)
    qkv = rng.normal(size=(B * T * 3 * C,))
    dout = rng.normal(size=(B * T * C,))
    out, att = oracle.attention_forward(qkv, B, T, C, NH)
    dqkv = oracle.attention_backward(dout, qkv, att, B, T, C, NH)
    qt = torch.tensor(qkv, requires_grad=True)
    HS = C // NH
    t = qt.view(B, T, 3, NH, HS)
    q, k, v = (t[:, :, i].transpose(1, 2) for i in range(3))
    y = F.scaled_dot_product_attention(q, k, v, is_causal=True).transpose(1, 2).reshape(-1)
    y.backward(torch.tensor(dout))
    np.testing.assert_allclose(dqkv, qt.grad.numpy(), rtol=1e-9, atol=1e-12)


def test_encoder_forward_is_a_gather_add():
    B, T, C, V = 2, 5, 8, 11
    rng = np.random.default_rng(5)
    wte = rng.normal(size=(V, C))
    wpe = rng.normal(size=(T, C))
    tok = rng.integers(0, V, size=(B, T)).astype(np.int32)
    out = oracle.encoder_forward(tok, wte, wpe, B, T, C).reshape(B, T, C)
    np.testing.assert_array_equal(out, wte[tok] + wpe[None])


# --------------------------------------------------------------------------
# AdamW


def test_adamw_matches_torch_adamw():
    rng = np.random.default_rng(6)
    n = 1000
    p0 = rng.normal(size=n)
    grads = [rng.normal(size=n) * 10 ** rng.uniform(-6, 0, size=n) for _ in range(3)]
    p = p0.copy()
    m = np.zeros(n)
    v = np.zeros(n)
    pt = torch.tensor(p0, requires_grad=True)
    opt = torch.optim.AdamW([pt], lr=6e-4, betas=(0.9, 0.95), eps=1e-8, weight_decay=0.1)
    for t, g in enumerate(grads, start=1):
        oracle.adamw(p, g, m, v, 6e-4, 0.9, 0.95, 1e-8, 0.1, t)
        pt.grad = torch.tensor(g)
        opt.step()
    np.testing.assert_allclose(p, pt.detach().numpy(), rtol=1e-12, atol=1e-15)


def test_adamw_first_step_closed_form():
    g = np.array([1e-3, -2.0, 5e-7, 0.0, -3e-9])
    p = np.ones_like(g)
    m = np.zeros_like(g)
    v = np.zeros_like(g)
    oracle.adamw(p, g, m, v, 1e-3, 0.9, 0.999, 1e-8, 0.0, 1)
    np.testing.assert_allclose(p, 1.0 - 1e-3 * g / (np.abs(g) + 1e-8), rtol=1e-12, atol=0)


# --------------------------------------------------------------------------
# whole model


def _torch_gpt2_loss(params, tok, tgt, d, B, T):
    """GPT-2 forward composed from torch.nn.functional routines (float64)."""
    sizes = inputs.param_sizes(d)
    ts = {}
    off = 0
    for name, s in zip(inputs.PARAM_NAMES, sizes):
        ts[name] = params[off:off + s]
        off += s
    C, L, NH = d.C, d.L, d.NH
    wte = ts["wte"].view(d.Vp, C)
    x = wte[tok] + ts["wpe"].view(d.maxT, C)[:T][None]
    for l in range(L):
        def sl(name, *shape):
            n = int(np.prod(shape))
            return ts[name][l * n:(l + 1) * n].view(*shape)
        h = F.layer_norm(x, (C,), sl("ln1w", C), sl("ln1b", C), eps=1e-5)
        qkv = F.linear(h, sl("qkvw", 3 * C, C), sl("qkvb", 3 * C))
        q, k, v = qkv.view(B, T, 3, NH, C // NH).unbind(2)
        a = F.scaled_dot_product_attention(q.transpose(1, 2), k.transpose(1, 2), v.transpose(1, 2),
                                           is_causal=True).transpose(1, 2).reshape(B, T, C)
        x = x + F.linear(a, sl("attprojw", C, C), sl("attprojb", C))
        h = F.layer_norm(x, (C,), sl("ln2w", C), sl("ln2b", C), eps=1e-5)
        h = F.gelu(F.linear(h, sl("fcw", 4 * C, C), sl("fcb", 4 * C)), approximate="tanh")
        x = x + F.linear(h, sl("fcprojw", C, 4 * C), sl("fcprojb", C))
    x = F.layer_norm(x, (C,), ts["lnfw"], ts["lnfb"], eps=1e-5)
    logits = F.linear(x, wte)[..., :d.V]
    return F.cross_entropy(logits.reshape(B * T, d.V), tgt.reshape(-1).long(), reduction="none")


def test_model_forward_backward_matches_torch_autograd():
    d = TINY
    B, T = 2, 32
    params = inputs.gpt2_params(d, seed=11, perturb=True).astype(np.float64)
    tok = inputs.tokens(11, 1, B, T, d.V)
    tgt = inputs.tokens(11, 2, B, T, d.V)
    m = _tiny_model(B, T)
    loss = m.forward(params, tok, tgt)
    grads = np.zeros_like(params)
    m.backward(grads)
    pt = torch.tensor(params, requires_grad=True)
    losses = _torch_gpt2_loss(pt, torch.tensor(tok).long(), torch.tensor(tgt), d, B, T)
    losses.mean().backward()
    np.testing.assert_allclose(m.act("losses"), losses.detach().numpy(), rtol=1e-11)
    assert abs(loss - losses.mean().item()) < 1e-11 * abs(loss)
    g = pt.grad.numpy()
    # the padded wte rows receive no gradient in either
    np.testing.assert_allclose(grads, g, rtol=1e-7, atol=1e-13)


def test_model_gradients_central_finite_differences():
    d = TINY
    B, T = 1, 12
    params = inputs.gpt2_params(d, seed=5, perturb=True).astype(np.float64)
    tok = inputs.tokens(5, 1, B, T, d.V)
    tgt = inputs.tokens(5, 2, B, T, d.V)
    m = _tiny_model(B, T)
    m.forward(params, tok, tgt)
    grads = np.zeros_like(params)
    m.backward(grads)
    rng = np.random.default_rng(7)
    offs = np.cumsum([0] + inputs.param_sizes(d))
    h = 1e-5
    for ti in range(16):
        lo, hi = offs[ti], offs[ti + 1]
        if ti == 0:  # wte: sample rows that are used as tokens, targets, and others
            rows = list(tok.reshape(-1)[:2]) + [int(rng.integers(0, d.V))]
            idxs = [lo + r * d.C + int(rng.integers(0, d.C)) for r in rows]
        elif ti == 1:  # wpe: only positions < T receive gradient
            idxs = [lo + t * d.C + int(rng.integers(0, d.C)) for t in (0, T - 1)]
        else:
            idxs = [int(i) for i in rng.integers(lo, hi, size=3)]
        for i in idxs:
            p = params.copy()
            p[i] += h
            lp = m.forward(p, tok, tgt)
            p[i] -= 2 * h
            lm = m.forward(p, tok, tgt)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - grads[i]) <= 1e-6 * max(abs(grads[i]), 1e-4), (ti, i, fd, grads[i])
    # positions >= T never reach the loss
    assert np.all(grads[offs[1] + T * d.C: offs[2]] == 0.0)


def test_loss_at_init_is_near_log_vocab():
    for d, B, T in ((TINY, 2, 32),):
        params = inputs.gpt2_params(d, seed=1337).astype(np.float64)
        tok = inputs.tokens(42, 1, B, T, d.V)
        tgt = inputs.tokens(42, 2, B, T, d.V)
        loss = _tiny_model(B, T, d).forward(params, tok, tgt)
        assert abs(loss - math.log(d.V)) < 0.3


def test_probabilities_sum_to_one_and_padding_is_masked():
    d = inputs.GPT2Dims(L=1, C=32, NH=2, V=50, Vp=64, maxT=16)
    B, T = 2, 16
    params = inputs.gpt2_params(d, seed=3, perturb=True).astype(np.float64)
    tok = inputs.tokens(3, 1, B, T, d.V)
    tgt = inputs.tokens(3, 2, B, T, d.V)
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    m.forward(params, tok, tgt)
    probs = m.act("probs").reshape(B * T, d.Vp)
    np.testing.assert_allclose(probs.sum(-1), 1.0, atol=1e-12)
    assert np.all(probs[:, d.V:] == 0)
    dl = m.act("dlogits").reshape(B * T, d.Vp)
    assert np.all(dl[:, d.V:] == 0)
    # each dlogits row sums to zero (probabilities minus a one-hot), scaled by 1/(B*T)
    np.testing.assert_allclose(dl.sum(-1), 0.0, atol=1e-15)
    att = m.act("att").reshape(B, d.NH, T, T)
    np.testing.assert_allclose(att.sum(-1), 1.0, atol=1e-12)
    # cross-entropy matches torch on the real columns
    logits = m.act("logits").reshape(B * T, d.Vp)[:, :d.V]
    ref = F.cross_entropy(torch.tensor(logits), torch.tensor(tgt.reshape(-1)).long(), reduction="none")
    np.testing.assert_allclose(m.act("losses"), ref.numpy(), rtol=1e-12)


def test_causal_mask_future_tokens_do_not_change_past():
    d = TINY
    B, T = 2, 32
    params = inputs.gpt2_params(d, seed=9, perturb=True).astype(np.float64)
    tok = inputs.tokens(9, 1, B, T, d.V)
    tgt = inputs.tokens(9, 2, B, T, d.V)
    m = _tiny_model(B, T)
    m.forward(params, tok, tgt)
    l0 = m.act("losses").reshape(B, T).copy()
    cut = 10
    tok2 = tok.copy()
    tok2[:, cut + 1:] = (tok2[:, cut + 1:] + 7) % d.V
    m.forward(params, tok2, tgt)
    l1 = m.act("losses").reshape(B, T)
    np.testing.assert_array_equal(l0[:, :cut + 1], l1[:, :cut + 1])
    assert np.any(l0[:, cut + 1:] != l1[:, cut + 1:])


def test_gradient_accumulation_equals_double_batch():
    d = TINY
    B, T = 2, 16
    params = inputs.gpt2_params(d, seed=21, perturb=True).astype(np.float64)
    tok = inputs.tokens(21, 1, 2 * B, T, d.V)
    tgt = inputs.tokens(21, 2, 2 * B, T, d.V)
    m = _tiny_model(B, T)
    acc = np.zeros_like(params)
    l_a = m.forward(params, tok[:B], tgt[:B], grad_accum_k=2)
    m.backward(acc)
    l_b = m.forward(params, tok[B:], tgt[B:], grad_accum_k=2)
    m.backward(acc)
    big = _tiny_model(2 * B, T)
    g2 = np.zeros_like(params)
    l_ab = big.forward(params, tok, tgt)
    big.backward(g2)
    assert abs((l_a + l_b) / 2 - l_ab) < 1e-12
    np.testing.assert_allclose(acc, g2, rtol=1e-9, atol=1e-15)


def test_zero_layers_is_bigram_softmax_regression():
    d = inputs.GPT2Dims(L=0, C=16, NH=2, V=40, Vp=48, maxT=8)
    B, T = 3, 8
    params = inputs.gpt2_params(d, seed=4, perturb=True).astype(np.float64)
    tok = inputs.tokens(4, 1, B, T, d.V)
    tgt = inputs.tokens(4, 2, B, T, d.V)
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    m.forward(params, tok, tgt)
    ts = m.split(params)
    wte = ts["wte"].reshape(d.Vp, d.C)
    x = wte[tok] + ts["wpe"].reshape(d.maxT, d.C)[None, :T]
    x = F.layer_norm(torch.tensor(x), (d.C,), torch.tensor(ts["lnfw"]), torch.tensor(ts["lnfb"]), eps=1e-5)
    logits = x.numpy() @ wte[:d.V].T
    ref = F.cross_entropy(torch.tensor(logits.reshape(-1, d.V)), torch.tensor(tgt.reshape(-1)).long(),
                          reduction="none")
    np.testing.assert_allclose(m.act("losses"), ref.numpy(), rtol=1e-12)


# --------------------------------------------------------------------------
# fused Linear + bias + GELU(tanh) + row softmax


def test_fused_op_matches_torch_composition():
    x, W, b = inputs.fused_op_inputs(7, 40, 33, seed=1)
    y = oracle.fused_linear_bias_gelu_softmax(x, W, b)
    ref = torch.softmax(F.gelu(F.linear(torch.tensor(x, dtype=torch.float64),
                                        torch.tensor(W, dtype=torch.float64),
                                        torch.tensor(b, dtype=torch.float64)),
                               approximate="tanh"), dim=1)
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(y.sum(1), 1.0, atol=1e-13)


def test_fused_op_zero_weight_is_softmax_of_gelu_bias():
    rng = np.random.default_rng(8)
    b = rng.uniform(-0.1, 0.1, size=29)
    x = rng.normal(size=(4, 12))
    y = oracle.fused_linear_bias_gelu_softmax(x, np.zeros((29, 12)), b)
    g = 0.5 * b * (1 + np.tanh(math.sqrt(2 / math.pi) * (b + 0.044715 * b ** 3)))
    e = np.exp(g - g.max())
    np.testing.assert_allclose(y, np.broadcast_to(e / e.sum(), y.shape), rtol=1e-13)


# --------------------------------------------------------------------------
# input generator


def test_input_generator_statistics_and_determinism():
    n = inputs.normal(7, 3, 200000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1.0) < 0.01
    np.testing.assert_array_equal(n, inputs.normal(7, 3, 200000))
    t = inputs.tokens(1, 1, 4, 1000, 50257)
    assert t.min() >= 0 and t.max() < 50257
    p = inputs.gpt2_params(TINY, 1337)
    s = inputs.param_sizes(TINY)
    wte = p[:s[0]].reshape(TINY.Vp, TINY.C)
    assert abs(wte.std() - 0.02) < 0.002
    r = inputs.round_to_bf16(np.array([1.0, 1.00390625, 1.01171875, -3.14159], dtype=np.float32))
    np.testing.assert_array_equal(r, torch.tensor([1.0, 1.00390625, 1.01171875, -3.14159]).bfloat16().float().numpy())
