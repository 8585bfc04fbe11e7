"""bf16 AdamW without master weights, with stochastic rounding (llm.c
"train_gpt2.cu", adamw_kernel3's branch for use_master_weights = 0), through
the C ABI against the oracle:
  - bit for bit equal to the oracle's float update + SquirrelNoise5 rounding,
    with the per-update seeds drawn from the page's xorshift* stream;
  - every new parameter is one of the two bf16 neighbours of the float64 update;
  - over many seeds the mean of the rounded parameters is the update itself;
  - CUDA-graph replays of the whole step equal eager steps bit for bit.
"""
import numpy as np
import pytest

import oracle
from transformer_lm_gb300 import gpt2 as G
from transformer_lm_gb300 import inputs

pytestmark = pytest.mark.gpu

D = inputs.GPT2Dims(L=2, C=128, NH=2, V=1000, Vp=1024, maxT=128)
HP = (1e-3, 0.9, 0.95, 1e-8, 0.1)


def _bits(x):
    return (np.ascontiguousarray(x, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _vals(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _case(seed):
    p = inputs.round_to_bf16(inputs.gpt2_params(D, seed, perturb=True)).astype(np.float32)
    n = p.size
    grads = [inputs.round_to_bf16(inputs.normal(seed, 10 + s, n, 1e-3)
                                  * np.exp(inputs.normal(seed, 20 + s, n, 1.0))).astype(np.float32)
             for s in range(3)]
    return p, grads


def _init(p):
    G.gpt2_init(D.L, D.C, D.NH, D.V, D.Vp, D.maxT, 1)
    G.gpt2_set_params(p)
    G.gpt2_set_master_weights(False)


def test_adamw_without_master_matches_oracle_bit_for_bit():
    p, grads = _case(3)
    _init(p)
    with pytest.raises(G.GPT2Error):
        G.gpt2_get_master()
    ref = _bits(p)
    m32 = np.zeros(p.size, np.float32)
    v32 = np.zeros(p.size, np.float32)
    rng = oracle.Rng(13371337)  # the model's stream at gpt2_init
    for t, g in enumerate(grads, start=1):
        G.gpt2_set_grads(g)
        G.gpt2_adamw(*HP, t)
        oracle.adamw_bf16_sr(ref, _bits(g), m32, v32, *HP, t, rng.u32())
        got = _bits(G.gpt2_get_params())
        diff = np.flatnonzero(got != ref)
        assert diff.size == 0, (t, diff[:5], got[diff[:5]], ref[diff[:5]])
    # float64 AdamW from the same bf16 start: each result is one of its two bf16 neighbours
    G.gpt2_set_params(p)
    G.gpt2_set_grads(grads[0])
    G.gpt2_adamw(*HP, 1)
    got = G.gpt2_get_params().astype(np.float64)
    p64 = p.astype(np.float64)
    oracle.adamw(p64, grads[0].astype(np.float64), np.zeros(p.size), np.zeros(p.size), *HP, 1)
    lo = _vals(_bits(p64.astype(np.float32)))
    hi = _vals(_bits(p64.astype(np.float32)) + 1)
    lo, hi = np.minimum(lo, hi).astype(np.float64), np.maximum(lo, hi).astype(np.float64)
    tol = 4 * np.abs(p64) * 2.0 ** -24
    assert np.all((got >= lo - tol) & (got <= hi + tol))
    G.gpt2_free()


def test_adamw_without_master_is_unbiased_over_seeds():
    p, grads = _case(4)
    _init(p)
    reps = 300
    acc = np.zeros(p.size)
    for _ in range(reps):  # each update draws a new seed from the model's stream
        G.gpt2_set_params(p)  # also clears the moments
        G.gpt2_set_grads(grads[0])
        G.gpt2_adamw(*HP, 1)
        acc += G.gpt2_get_params()
    G.gpt2_free()
    mean = acc / reps
    p64 = p.astype(np.float64)
    oracle.adamw(p64, grads[0].astype(np.float64), np.zeros(p.size), np.zeros(p.size), *HP, 1)
    b = _bits(p64.astype(np.float32))
    ulp = np.abs(_vals(b + 1).astype(np.float64) - _vals(b).astype(np.float64))
    # each element within 6 standard errors of a Bernoulli over one ulp
    err = np.abs(mean - p64)
    assert np.all(err <= 6 * 0.5 * ulp / np.sqrt(reps) + 4 * np.abs(p64) * 2.0 ** -24)
    # no systematic bias across elements (round-to-nearest would leave up to 1/2 ulp each)
    z = (mean - p64) / ulp
    assert abs(z.mean()) < 0.01, z.mean()


def test_train_step_graph_replays_without_master_match_eager_steps():
    import torch
    p, _ = _case(5)
    B, T = 2, 64
    batches = [(inputs.tokens(5, 2 * i + 1, B, T, D.V), inputs.tokens(5, 2 * i + 2, B, T, D.V))
               for i in range(4)]
    dt = torch.zeros(B * T, dtype=torch.int32, device="cuda")
    dg = torch.zeros(B * T, dtype=torch.int32, device="cuda")
    dl = torch.zeros(1, device="cuda")

    def run(use_graph):
        _init(p)
        losses = []
        for i, (tok, tgt) in enumerate(batches):
            dt.copy_(torch.from_numpy(tok.reshape(-1)))
            dg.copy_(torch.from_numpy(tgt.reshape(-1)))
            if use_graph:
                G.gpt2_train_step(dt, dg, B, T, *HP, i + 1, dl)
            else:
                G.gpt2_forward_device(dt, dg, B, T, dl)
                G.gpt2_zero_grad()
                G.gpt2_backward()
                G.gpt2_adamw(*HP, i + 1)
            G.gpt2_sync()
            losses.append(float(dl.item()))
        out = (losses, G.gpt2_get_params())
        G.gpt2_free()
        return out

    l_e, p_e = run(False)
    l_g, p_g = run(True)
    assert l_e == l_g
    assert np.array_equal(p_e, p_g)


def test_master_weights_can_be_turned_back_on():
    p, grads = _case(6)
    _init(p)
    G.gpt2_set_master_weights(True)
    assert np.array_equal(G.gpt2_get_master(), G.gpt2_get_params())
    G.gpt2_free()
    G.gpt2_init_ex(2, 64, 4, 512, 512, 32, 1, G.GPT2_FP32, 0)
    with pytest.raises(G.GPT2Error) as e:
        G.gpt2_set_master_weights(False)
    assert e.value.code == -1
    G.gpt2_free()
