"""Forward-only inference through the C ABI (llm.c "train_gpt2.cu":
fused_classifier_kernel3's probs output, sample_softmax, and the generation
block of main), against the oracle:
  - probabilities after a forward without targets: softmax over the first V
    logits, zero on the padding, rows summing to one;
  - gpt2_sample: the oracle's sample_softmax on the same logits, for many coins
    (where a coin falls within rounding distance of a cumulative-probability
    boundary, either neighbouring index is accepted);
  - gpt2_generate: equal to stepping forward + sample by hand with the page's
    xorshift* coins, and (fp32) to the oracle's own forward + sampling.
"""
import numpy as np
import pytest

import oracle
from transformer_lm_gb300 import gpt2 as G
from transformer_lm_gb300 import inputs

pytestmark = pytest.mark.gpu

SMALL_BF16 = inputs.GPT2Dims(L=2, C=128, NH=2, V=1000, Vp=1024, maxT=64)


def _init(d, prec, tc, params):
    G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, prec, tc)
    G.gpt2_set_params(params)


def _softmax64(lg):
    e = np.exp(lg - lg.max())
    return e / e.sum()


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_probs_after_forward_without_targets(prec):
    d = inputs.TINY if prec == "fp32" else SMALL_BF16
    B, T = 2, 32
    params = inputs.gpt2_params(d, 21, perturb=True)
    if prec == "bf16":
        params = inputs.round_to_bf16(params)
        _init(d, G.GPT2_BF16, 1, params)
    else:
        _init(d, G.GPT2_FP32, 0, params)
    tok = inputs.tokens(21, 1, B, T, d.V)
    assert G.gpt2_forward(tok, None, B, T) == -1.0
    probs = G.gpt2_get_activation("probs").reshape(B * T, d.Vp).astype(np.float64)
    logits = G.gpt2_get_activation("logits").reshape(B * T, d.Vp).astype(np.float64)
    G.gpt2_free()
    assert np.all(probs[:, d.V:] == 0)
    np.testing.assert_allclose(probs.sum(1), 1.0, atol=1e-5)
    # the kernel's softmax of its own logits
    ref_own = np.stack([_softmax64(r[:d.V]) for r in logits])
    np.testing.assert_allclose(probs[:, :d.V], ref_own, rtol=1e-5, atol=1e-9)
    # the oracle's probabilities
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    m.forward(params.astype(np.float64), tok, None)
    ref = m.act("probs").reshape(B * T, d.Vp)
    if prec == "fp32":
        np.testing.assert_allclose(probs, ref, rtol=1e-4, atol=1e-9)
    else:
        tv = 0.5 * np.abs(probs - ref).sum(1)  # total variation distance per row
        assert tv.max() < 0.05, tv.max()


def _check_sample(idx, row, coin):
    """idx must be the oracle's sample_softmax index, or (within rounding of a
    cumulative boundary) a neighbour whose interval touches the coin."""
    want = oracle.sample_softmax(row, coin)
    if idx == want:
        return True
    cdf = np.cumsum(_softmax64(row))
    lo = cdf[idx - 1] if idx > 0 else 0.0
    return abs(idx - want) == 1 and (abs(coin - lo) < 1e-5 or abs(coin - cdf[idx]) < 1e-5)


@pytest.mark.parametrize("prec", ["fp32", "bf16"])
def test_sample_matches_oracle_sample_softmax(prec):
    d = inputs.TINY if prec == "fp32" else SMALL_BF16
    B, T = 2, 32
    params = inputs.gpt2_params(d, 22, perturb=True)
    if prec == "bf16":
        params = inputs.round_to_bf16(params)
        _init(d, G.GPT2_BF16, 1, params)
    else:
        _init(d, G.GPT2_FP32, 0, params)
    tok = inputs.tokens(22, 1, B, T, d.V)
    G.gpt2_forward(tok, None, B, T)
    logits = G.gpt2_get_activation("logits").reshape(B, T, d.Vp).astype(np.float64)
    rng = np.random.default_rng(22)
    for t in (0, 7, T - 1):
        for _ in range(100):
            coins = rng.random(B).astype(np.float32)
            got = G.gpt2_sample(t, coins)
            for b in range(B):
                assert _check_sample(int(got[b]), logits[b, t, :d.V], float(coins[b])), (t, b, coins[b])
    # a coin of 0 gives the first index with non-zero probability; sharp rows give their argmax
    got = G.gpt2_sample(3, np.zeros(B, np.float32))
    assert np.all(got == 0)
    with pytest.raises(G.GPT2Error):
        G.gpt2_sample(T, np.zeros(B, np.float32))
    with pytest.raises(G.GPT2Error):
        G.gpt2_sample(0, np.ones(B, np.float32))
    G.gpt2_forward(tok, tok, B, T)
    with pytest.raises(G.GPT2Error) as e:
        G.gpt2_sample(0, np.zeros(B, np.float32))  # logits were overwritten by the backward seed
    assert e.value.code == -2
    G.gpt2_free()


def test_generate_equals_forward_and_sample_step_by_step():
    d = SMALL_BF16
    B, T = 3, 24
    params = inputs.round_to_bf16(inputs.gpt2_params(d, 23, perturb=True))
    start = np.zeros((B, T), dtype=np.int32)
    start[:, 0] = [5, 77, 999]
    _init(d, G.GPT2_BF16, 1, params)
    gen, st = G.gpt2_generate(start, B, T, 1, T, 1337)
    G.gpt2_free()
    # by hand: the same forward and sampler, the page's coins
    _init(d, G.GPT2_BF16, 1, params)
    tok = start.copy()
    rng = oracle.Rng(1337)
    for t in range(1, T):
        G.gpt2_forward(tok, None, B, T)
        coins = np.array([rng.f32() for _ in range(B)], dtype=np.float32)
        tok[:, t] = G.gpt2_sample(t - 1, coins)
    G.gpt2_free()
    assert np.array_equal(gen, tok)
    assert st == rng.state.value
    assert np.array_equal(gen[:, 0], start[:, 0])


def test_generate_fp32_agrees_with_oracle():
    """fp32 model: the oracle's float64 forward and sample_softmax with the same
    coins pick the same tokens (until a coin lands within rounding distance of
    a cumulative boundary, after which the continuations may differ)."""
    d = inputs.TINY
    B, T = 2, 20
    params = inputs.gpt2_params(d, 24, perturb=True)
    start = np.zeros((B, T), dtype=np.int32)
    start[:, 0] = [3, 300]
    _init(d, G.GPT2_FP32, 0, params)
    gen, _ = G.gpt2_generate(start, B, T, 1, T, 1337)
    G.gpt2_free()
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    p64 = params.astype(np.float64)
    tok = start.copy()
    rng = oracle.Rng(1337)
    agree = 0
    for t in range(1, T):
        m.forward(p64, tok, None)
        logits = m.act("logits").reshape(B, T, d.Vp)
        coins = [rng.f32() for _ in range(B)]
        near = False
        for b in range(B):
            row = logits[b, t - 1, :d.V]
            tok[b, t] = oracle.sample_softmax(row, coins[b])
            cdf = np.cumsum(_softmax64(row))
            near |= bool(np.min(np.abs(cdf - coins[b])) < 1e-6)
        if near:
            break
        assert np.array_equal(gen[:, t], tok[:, t]), t
        agree += 1
    assert agree >= 10
