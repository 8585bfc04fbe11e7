"""fp16 training (llm.c "train_gpt2.cu", the ENABLE_FP16 build: floatX = half)
with dynamic loss scaling, through the C ABI against the oracle:
  - the GEMM (every operand layout and epilogue, split-K), causal attention and
    LayerNorm kernels with fp16 operands against the oracle;
  - one training step: loss within 2e-2, per-tensor gradient cosine >= 0.99
    (the mixed-precision bounds), master weights after AdamW;
  - the loss scaler: an overflowing step is skipped (parameters and moments
    unchanged) and halves the scale; growth_interval clean steps double it;
  - CUDA-graph replays equal eager steps bit for bit, scaler state included.
Inputs are rounded to fp16 first, so both sides start from identical values.
"""
import numpy as np
import pytest

import oracle
from transformer_lm_gb300 import gpt2 as G
from transformer_lm_gb300 import inputs
from tests.gpu_util import cosine, dev, empty, host, rel_to_max

pytestmark = pytest.mark.gpu

r16 = inputs.round_to_fp16


def _operands(M, N, K, seed):
    A = inputs.normal(seed, 1, M * K).reshape(M, K).astype(np.float32)
    B = inputs.normal(seed, 2, N * K, 0.05).reshape(N, K).astype(np.float32)
    bias = inputs.normal(seed, 3, N, 0.5).astype(np.float32)
    aux = inputs.normal(seed, 4, M * N).reshape(M, N).astype(np.float32)
    D0 = inputs.normal(seed, 5, M * N, 0.3).reshape(M, N).astype(np.float32)
    return tuple(r16(x) for x in (A, B, bias, aux, D0))


def _stored(X, kmajor):
    S = X if kmajor else X.T
    ld = (S.shape[1] + 7) // 8 * 8
    P = np.zeros((S.shape[0], ld), dtype=np.float32)
    P[:, :S.shape[1]] = S
    return P, ld


@pytest.mark.parametrize("tc", [1, 0])
@pytest.mark.parametrize("a_km,b_km", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("shape", [(200, 136, 72), (130, 264, 1000), (1024, 768, 768), (512, 520, 136)],
                         ids=lambda s: "x".join(map(str, s)))
def test_fp16_gemm_layouts_match_oracle(tc, a_km, b_km, shape):
    M, N, K = shape
    A, B, bias, aux, D0 = _operands(M, N, K, 7 + M + N + K)
    ref = oracle.matmul_forward(A, B, bias)
    sA, lda = _stored(A, a_km)
    sB, ldb = _stored(B, b_km)
    D = empty((M, N), "f16")
    G.gpt2_gemm(G.GPT2_FP16, tc, "store", dev(sA, "f16"), lda, a_km, dev(sB, "f16"), ldb, b_km, D, N,
                bias=dev(bias, "f16"), M=M, N=N, K=K)
    G.gpt2_device_status()
    assert rel_to_max(host(D), ref) < 2e-3


@pytest.mark.parametrize("epi", ["gelu", "resid", "gelu_bwd", "accum"])
@pytest.mark.parametrize("shape", [(300, 392, 200), (2048, 264, 520)], ids=lambda s: "x".join(map(str, s)))
def test_fp16_gemm_epilogues_match_oracle(epi, shape):
    M, N, K = shape
    A, B, bias, aux, D0 = _operands(M, N, K, 99)
    acc = oracle.matmul_forward(A, B, None)
    ref2 = None
    if epi == "gelu":
        ref = acc + bias
        ref2 = oracle.gelu_forward(ref)
    elif epi == "resid":
        ref = acc + bias + aux
    elif epi == "gelu_bwd":
        ref = oracle.gelu_backward(aux, acc)
    else:
        ref = D0.astype(np.float64) + acc
    D = dev(D0, "f16") if epi == "accum" else empty((M, N), "f16")
    D2 = empty((M, N), "f16") if epi == "gelu" else None
    G.gpt2_gemm(G.GPT2_FP16, 1, epi, dev(A, "f16"), K, 1, dev(B.T, "f16"), N, 0, D, N,
                bias=dev(bias, "f16"), aux=dev(aux, "f16"), ldaux=N, D2=D2, M=M, N=N, K=K)
    G.gpt2_device_status()
    assert rel_to_max(host(D), ref) < 3e-3
    if D2 is not None:
        assert rel_to_max(host(D2), ref2) < 3e-3


def test_fp16_gemm_split_k_accumulate_matches_oracle():
    import torch
    M, N, K = 768, 768, 8192
    A, B, bias, aux, D0 = _operands(M, N, K, 21)
    ref = D0.astype(np.float64) + oracle.matmul_forward(A, B, None)
    sA, lda = _stored(A, 0)
    sB, ldb = _stored(B, 0)
    ws = torch.empty(16 * M * N + 64, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):
        D = dev(D0, "f16")
        G.gpt2_gemm(G.GPT2_FP16, 1, "accum", dev(sA, "f16"), lda, 0, dev(sB, "f16"), ldb, 0, D, N,
                    M=M, N=N, K=K, ws=ws, ws_floats=ws.numel())
        G.gpt2_device_status()
        outs.append(host(D))
    assert rel_to_max(outs[0], ref) < 2e-3
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("B,T,C,NH,tc", [(2, 64, 128, 2, 1), (2, 130, 128, 2, 1), (3, 17, 128, 2, 1),
                                         (2, 256, 256, 4, 1), (1, 40, 64, 2, 0)])
def test_fp16_attention_forward_backward_match_oracle(B, T, C, NH, tc):
    import torch
    qkv = r16(inputs.normal(5 + T, 1, B * T * 3 * C).astype(np.float32))
    dout = r16(inputs.normal(5 + T, 2, B * T * C, 0.1).astype(np.float32))
    ref_out, att = oracle.attention_forward(qkv, B, T, C, NH)
    ref_dqkv = oracle.attention_backward(dout, qkv, att, B, T, C, NH)
    d_qkv = dev(qkv, "f16")
    out = empty((B * T * C,), "f16")
    lse = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_forward(G.GPT2_FP16, tc, d_qkv, out, lse, B, T, C, NH)
    dqkv = empty((B * T * 3 * C,), "f16")
    Dsc = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_backward(G.GPT2_FP16, tc, dev(dout, "f16"), d_qkv, out, lse, dqkv, Dsc, B, T, C, NH)
    G.gpt2_device_status()
    assert rel_to_max(host(out), ref_out) < 4e-3
    got = host(dqkv).reshape(B, T, 3, C)
    ref = ref_dqkv.reshape(B, T, 3, C)
    for part in range(3):
        assert rel_to_max(got[:, :, part], ref[:, :, part]) < 8e-3, part


@pytest.mark.parametrize("N,C", [(1000, 768), (8192, 768), (300, 1024), (515, 640), (9, 256)])
def test_fp16_layernorm_forward_backward_match_oracle(N, C):
    import torch
    x = r16(inputs.normal(N + C, 1, N * C, 2.0).reshape(N, C).astype(np.float32) + 0.5)
    w = r16((1.0 + inputs.normal(N + C, 2, C, 0.1)).astype(np.float32))
    b = r16(inputs.normal(N + C, 3, C, 0.1).astype(np.float32))
    dy = r16(inputs.normal(N + C, 4, N * C, 0.01).reshape(N, C).astype(np.float32))
    d0 = r16(inputs.normal(N + C, 5, N * C, 0.01).reshape(N, C).astype(np.float32))
    ref, mean, rstd = oracle.layernorm_forward(x, w, b)
    out = empty((N, C), "f16")
    dmean = torch.zeros(N, device="cuda")
    drstd = torch.zeros(N, device="cuda")
    dx = dev(x, "f16")
    G.gpt2_layernorm_forward(G.GPT2_FP16, out, dmean, drstd, dx, dev(w, "f16"), dev(b, "f16"), N, C)
    assert rel_to_max(host(out), ref) < 2e-3
    np.testing.assert_allclose(host(drstd), rstd, rtol=1e-4)
    dinp = d0.astype(np.float64).copy()
    dw = np.ones(C)
    db = np.ones(C)
    oracle.layernorm_backward(dinp, dw, db, dy, x, w, mean, rstd)
    g_dinp = dev(d0, "f16")
    g_dw = dev(np.ones(C, dtype=np.float32), "f16")
    g_db = dev(np.ones(C, dtype=np.float32), "f16")
    scratch = torch.zeros(G.gpt2_layernorm_backward_scratch_floats(C), device="cuda")
    G.gpt2_layernorm_backward(G.GPT2_FP16, g_dinp, g_dw, g_db, dev(dy, "f16"), dx, dev(w, "f16"), dmean,
                              drstd, N, C, 1, scratch)
    G.gpt2_device_status()
    assert rel_to_max(host(g_dinp), dinp) < 4e-3
    for got, want in ((host(g_dw), dw), (host(g_db), db)):
        # rounded once to fp16 near its value (a half ulp is 2^-11 relative)
        assert np.max(np.abs(got - want)) <= 2.0 ** -10 * np.max(np.abs(want)) + 4e-3 * np.max(np.abs(want - 1.0))


SMALL = inputs.GPT2Dims(L=2, C=128, NH=2, V=1000, Vp=1024, maxT=256)


def _split(flat, d):
    out, off = {}, 0
    for name, s in zip(inputs.PARAM_NAMES, inputs.param_sizes(d)):
        out[name] = flat[off:off + s]
        off += s
    return out


@pytest.mark.parametrize("tc", [1, 0])
def test_fp16_step_matches_oracle(tc):
    d = SMALL
    B, T = 2, 192
    params = r16(inputs.gpt2_params(d, 11, perturb=True))
    tok = inputs.tokens(11, 1, B, T, d.V)
    tgt = inputs.tokens(11, 2, B, T, d.V)
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    ref_loss = m.forward(params.astype(np.float64), tok, tgt)
    ref_g = np.zeros(params.size)
    m.backward(ref_g)
    G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, G.GPT2_FP16, tc)
    G.gpt2_set_params(params)
    assert np.array_equal(G.gpt2_get_params(), params)
    G.gpt2_set_loss_scaling(1024.0, 2000)
    G.gpt2_zero_grad()
    loss = G.gpt2_forward(tok, tgt, B, T)
    assert abs(loss - ref_loss) <= 2e-2, (loss, ref_loss)
    G.gpt2_backward()
    g = G.gpt2_get_grads()  # unscaled
    cos = {n: cosine(_split(g, d)[n], _split(ref_g, d)[n]) for n in inputs.PARAM_NAMES}
    print(f"fp16 tc={tc}: loss {loss:.6f} oracle {ref_loss:.6f}; grad cosines",
          {k: round(v, 6) for k, v in cos.items()})
    for n, c in cos.items():
        assert c >= 0.99, (n, c)
    G.gpt2_adamw(6e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    master = G.gpt2_get_master()
    ref_p = params.astype(np.float64)
    oracle.adamw(ref_p, ref_g, np.zeros_like(ref_p), np.zeros_like(ref_p), 6e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    band = np.abs(ref_g) < 1e-7  # exact zero gradients (key biases) move by noise/eps
    assert cosine((master - params)[~band], (ref_p - params)[~band]) >= 0.99
    assert G.gpt2_get_loss_scale() == (1024.0, 0)
    G.gpt2_free()


def test_fp16_loss_scaler_skips_overflow_and_adapts():
    d = SMALL
    B, T = 2, 64
    params = r16(inputs.gpt2_params(d, 12, perturb=True))
    tok = inputs.tokens(12, 1, B, T, d.V)
    tgt = inputs.tokens(12, 2, B, T, d.V)
    G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, G.GPT2_FP16, 1)
    G.gpt2_set_params(params)
    # a scale whose seeded dlogits (scale / (B T)) exceed the fp16 range
    G.gpt2_set_loss_scaling(2.0 ** 30, 2)
    G.gpt2_zero_grad()
    G.gpt2_forward(tok, tgt, B, T)
    G.gpt2_backward()
    G.gpt2_adamw(6e-4, 0.9, 0.95, 1e-8, 0.1, 1)
    assert np.array_equal(G.gpt2_get_params(), params)  # skipped
    assert np.array_equal(G.gpt2_get_master(), params)
    assert G.gpt2_get_loss_scale() == (2.0 ** 29, 1)
    # a safe scale: two clean steps double it
    G.gpt2_set_loss_scaling(256.0, 2)
    for step in (1, 2):
        G.gpt2_zero_grad()
        G.gpt2_forward(tok, tgt, B, T)
        G.gpt2_backward()
        G.gpt2_adamw(6e-4, 0.9, 0.95, 1e-8, 0.1, step)
        assert not np.array_equal(G.gpt2_get_master(), params)
    assert G.gpt2_get_loss_scale() == (512.0, 0)
    with pytest.raises(G.GPT2Error):
        G.gpt2_set_loss_scaling(1000.0, 2)  # not a power of two
    G.gpt2_free()
    G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, G.GPT2_BF16, 1)
    with pytest.raises(G.GPT2Error) as e:
        G.gpt2_set_loss_scaling(256.0, 2)
    assert e.value.code == -1
    assert G.gpt2_get_loss_scale() == (1.0, 0)
    G.gpt2_free()


def test_fp16_train_step_graph_replays_match_eager_steps():
    import torch
    d = SMALL
    B, T = 2, 128
    params = r16(inputs.gpt2_params(d, 14, perturb=True))
    batches = [(inputs.tokens(14, 2 * i + 1, B, T, d.V), inputs.tokens(14, 2 * i + 2, B, T, d.V))
               for i in range(4)]
    dt = torch.zeros(B * T, dtype=torch.int32, device="cuda")
    dg = torch.zeros(B * T, dtype=torch.int32, device="cuda")
    dl = torch.zeros(1, device="cuda")

    def run(use_graph):
        G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, G.GPT2_FP16, 1)
        G.gpt2_set_params(params)
        G.gpt2_set_loss_scaling(2.0 ** 12, 2)  # doubles during the run
        losses = []
        for i, (tok, tgt) in enumerate(batches):
            dt.copy_(torch.from_numpy(tok.reshape(-1)))
            dg.copy_(torch.from_numpy(tgt.reshape(-1)))
            if use_graph:
                G.gpt2_train_step(dt, dg, B, T, 6e-4, 0.9, 0.95, 1e-8, 0.1, i + 1, dl)
            else:
                G.gpt2_forward_device(dt, dg, B, T, dl)
                G.gpt2_zero_grad()
                G.gpt2_backward()
                G.gpt2_adamw(6e-4, 0.9, 0.95, 1e-8, 0.1, i + 1)
            G.gpt2_sync()
            losses.append(float(dl.item()))
        out = (losses, G.gpt2_get_params(), G.gpt2_get_master(), G.gpt2_get_loss_scale())
        G.gpt2_free()
        return out

    e, g = run(False), run(True)
    assert e[0] == g[0]
    assert np.array_equal(e[1], g[1]) and np.array_equal(e[2], g[2])
    assert e[3] == g[3] == (2.0 ** 14, 0)


def test_fp16_124m_step_matches_oracle():
    """GPT-2 124M in fp16 at B=2, T=256: every gradient tensor against the oracle."""
    d = inputs.GPT2_124M
    B, T = 2, 256
    params = r16(inputs.gpt2_params(d, 17))
    tok = inputs.tokens(17, 1, B, T, d.V)
    tgt = inputs.tokens(17, 2, B, T, d.V)
    G.gpt2_init_ex(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, 1, G.GPT2_FP16, 1)
    G.gpt2_set_params(params)
    G.gpt2_zero_grad()
    loss = G.gpt2_forward(tok, tgt, B, T)
    G.gpt2_backward()
    g = G.gpt2_get_grads()
    scale, skipped = G.gpt2_get_loss_scale()
    G.gpt2_free()
    assert np.all(np.isfinite(g)), "the default scale overflowed at this size"
    m = oracle.Model(d.L, d.C, d.NH, d.V, d.Vp, d.maxT, B, T)
    ref_loss = m.forward(params.astype(np.float64), tok, tgt)
    ref_g = np.zeros(params.size)
    m.backward(ref_g)
    assert abs(loss - ref_loss) <= 2e-2
    cos = {n: cosine(_split(g, d)[n], _split(ref_g, d)[n]) for n in inputs.PARAM_NAMES}
    print(f"fp16 124M B=2 T=256 (scale {scale}): grad cosines", {k: round(v, 6) for k, v in cos.items()})
    for n, c in cos.items():
        assert c >= 0.99, (n, c)
