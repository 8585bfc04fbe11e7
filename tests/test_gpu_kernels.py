"""Kernel-level parity against the oracle: every GEMM operand layout and
epilogue (tcgen05 bf16, SIMT fp32 and bf16), and causal attention forward and
backward (tensor-core flash kernels and SIMT), on shapes that span several
tiles and end in ragged tails."""
import numpy as np
import pytest

import oracle
from transformer_lm_gb300 import inputs
from transformer_lm_gb300 import gpt2 as G
from tests.gpu_util import dev, host, empty, rel_to_max, max_rel_floor

pytestmark = pytest.mark.gpu

# several tiles, ragged tails, and m-block counts that select 1, 2 and 4 CTAs per cluster
SHAPES = [(200, 136, 72), (256, 512, 128), (130, 264, 1000), (1024, 768, 768), (64, 8, 16),
          (512, 520, 136), (2048, 1032, 264)]


def _operands(M, N, K, seed, bf16):
    A = inputs.normal(seed, 1, M * K).reshape(M, K).astype(np.float32)
    B = inputs.normal(seed, 2, N * K, 0.05).reshape(N, K).astype(np.float32)
    bias = inputs.normal(seed, 3, N, 0.5).astype(np.float32)
    aux = inputs.normal(seed, 4, M * N).reshape(M, N).astype(np.float32)
    D0 = inputs.normal(seed, 5, M * N, 0.3).reshape(M, N).astype(np.float32)
    if bf16:
        A, B, bias, aux, D0 = (inputs.round_to_bf16(x) for x in (A, B, bias, aux, D0))
    return A, B, bias, aux, D0


def _ref(epi, A, B, bias, aux, D0):
    acc = oracle.matmul_forward(A, B, None)
    if epi == "store":
        return acc + bias, None
    if epi == "gelu":
        pre = acc + bias
        return pre, oracle.gelu_forward(pre)
    if epi == "resid":
        return acc + bias + aux, None
    if epi == "gelu_bwd":
        return oracle.gelu_backward(aux, acc), None
    if epi == "accum":
        return D0.astype(np.float64) + acc, None
    raise ValueError(epi)


MODES = [("bf16", 1), ("bf16", 0), ("f32", 0)]


def _stored(X, kmajor):
    """Storage of logical X[rows, K]: K-major = X itself, MN-major = X^T; the
    leading dimension is padded to a multiple of 8 elements (16 bytes)."""
    S = X if kmajor else X.T
    ld = (S.shape[1] + 7) // 8 * 8
    P = np.zeros((S.shape[0], ld), dtype=np.float32)
    P[:, :S.shape[1]] = S
    return P, ld


@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m[0]}-tc{m[1]}")
@pytest.mark.parametrize("a_km,b_km", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_gemm_layouts_match_oracle(mode, a_km, b_km, shape):
    dt, tc = mode
    M, N, K = shape
    bf16 = dt == "bf16"
    A, B, bias, aux, D0 = _operands(M, N, K, 7 + M + N + K, bf16)
    ref, _ = _ref("store", A, B, bias, aux, D0)
    sA, lda = _stored(A, a_km)
    sB, ldb = _stored(B, b_km)
    D = empty((M, N), dt)
    G.gpt2_gemm(G.GPT2_BF16 if bf16 else G.GPT2_FP32, tc, "store", dev(sA, dt), lda, a_km,
                dev(sB, dt), ldb, b_km, D, N, bias=dev(bias, dt), M=M, N=N, K=K)
    G.gpt2_device_status()
    err = rel_to_max(host(D), ref)
    assert err < (8e-3 if bf16 else 1e-5), err


@pytest.mark.parametrize("shape,a_km,b_km", [((768, 768, 8192), 0, 0), ((300, 264, 4096), 0, 0),
                                              ((1152, 384, 6144), 0, 0), ((520, 136, 3000), 1, 1)],
                         ids=lambda x: "x".join(map(str, x)) if isinstance(x, tuple) else str(x))
def test_gemm_split_k_accumulate_matches_oracle(shape, a_km, b_km):
    """D += A B^T for weight-gradient shapes (few output tiles, long K) with a
    scratch, so that K is split into ranges reduced in order; the result must
    match the oracle and repeat bit for bit."""
    import torch
    M, N, K = shape
    A, B, bias, aux, D0 = _operands(M, N, K, 21 + M + K, True)
    ref, _ = _ref("accum", A, B, bias, aux, D0)
    sA, lda = _stored(A, a_km)
    sB, ldb = _stored(B, b_km)
    dA, dB = dev(sA, "bf16"), dev(sB, "bf16")
    ws = torch.empty(16 * M * N + 64, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):
        D = dev(D0, "bf16")
        G.gpt2_gemm(G.GPT2_BF16, 1, "accum", dA, lda, a_km, dB, ldb, b_km, D, N, M=M, N=N, K=K,
                    ws=ws, ws_floats=ws.numel())
        G.gpt2_device_status()
        outs.append(host(D))
    assert rel_to_max(outs[0], ref) < 1e-2
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("shape,a_km,b_km", [((2048, 768, 12288), 1, 0), ((1024, 264, 16384), 1, 1),
                                              ((2048, 520, 16384), 0, 0), ((8192, 768, 6400), 1, 0)],
                         ids=lambda x: "x".join(map(str, x)) if isinstance(x, tuple) else str(x))
def test_gemm_split_k_store_matches_oracle(shape, a_km, b_km):
    """D = A B^T without bias over a long K with a scratch (the classifier's
    dlnf shape family): K may be split into ranges whose fp32 partials are
    summed in order and stored, so D's previous contents must not leak in; the
    result must match the oracle and repeat bit for bit."""
    import torch
    M, N, K = shape
    A, B, bias, aux, D0 = _operands(M, N, K, 31 + M + K, True)
    ref = oracle.matmul_forward(A, B, None)
    sA, lda = _stored(A, a_km)
    sB, ldb = _stored(B, b_km)
    dA, dB = dev(sA, "bf16"), dev(sB, "bf16")
    ws = torch.empty(3 * M * N + 64, dtype=torch.float32, device="cuda")
    outs = []
    for _ in range(2):
        D = dev(D0 * 1e3, "bf16")  # stale contents a += would keep
        G.gpt2_gemm(G.GPT2_BF16, 1, "store", dA, lda, a_km, dB, ldb, b_km, D, N, M=M, N=N, K=K,
                    ws=ws, ws_floats=ws.numel())
        G.gpt2_device_status()
        outs.append(host(D))
    assert rel_to_max(outs[0], ref) < 1e-2
    assert np.array_equal(outs[0], outs[1])


@pytest.mark.parametrize("mode", MODES, ids=lambda m: f"{m[0]}-tc{m[1]}")
@pytest.mark.parametrize("epi", ["gelu", "resid", "gelu_bwd", "accum"])
@pytest.mark.parametrize("shape", [(300, 392, 200), (1024, 392, 200), (2048, 264, 520)],
                         ids=lambda s: "x".join(map(str, s)))
def test_gemm_epilogues_match_oracle(mode, epi, shape):
    dt, tc = mode
    bf16 = dt == "bf16"
    M, N, K = shape
    A, B, bias, aux, D0 = _operands(M, N, K, 99, bf16)
    ref, ref2 = _ref(epi, A, B, bias, aux, D0)
    D = dev(D0, dt) if epi == "accum" else empty((M, N), dt)
    D2 = empty((M, N), dt) if epi == "gelu" else None
    G.gpt2_gemm(G.GPT2_BF16 if bf16 else G.GPT2_FP32, tc, epi, dev(A, dt), K, 1, dev(B.T, dt), N, 0,
                D, N, bias=dev(bias, dt), aux=dev(aux, dt), ldaux=N, D2=D2, M=M, N=N, K=K)
    G.gpt2_device_status()
    tol = 1e-2 if bf16 else 1e-5
    assert rel_to_max(host(D), ref) < tol
    if D2 is not None:
        assert rel_to_max(host(D2), ref2) < tol


@pytest.mark.parametrize("B,T,C,NH,dt,tc", [
    (2, 64, 128, 2, "bf16", 1), (2, 130, 128, 2, "bf16", 1), (1, 1, 128, 2, "bf16", 1),
    (2, 256, 256, 4, "bf16", 1), (3, 17, 128, 2, "bf16", 1),
    (2, 70, 64, 4, "f32", 0), (2, 33, 128, 2, "f32", 0), (1, 40, 64, 2, "bf16", 0)])
def test_attention_forward_backward_match_oracle(B, T, C, NH, dt, tc):
    bf16 = dt == "bf16"
    qkv = inputs.normal(5 + T, 1, B * T * 3 * C).astype(np.float32)
    dout = inputs.normal(5 + T, 2, B * T * C, 0.1).astype(np.float32)
    if bf16:
        qkv, dout = inputs.round_to_bf16(qkv), inputs.round_to_bf16(dout)
    ref_out, att = oracle.attention_forward(qkv, B, T, C, NH)
    ref_dqkv = oracle.attention_backward(dout, qkv, att, B, T, C, NH)
    prec = G.GPT2_BF16 if bf16 else G.GPT2_FP32
    d_qkv = dev(qkv, dt)
    out = empty((B * T * C,), dt)
    import torch
    lse = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_forward(prec, tc, d_qkv, out, lse, B, T, C, NH)
    dqkv = empty((B * T * 3 * C,), dt)
    Dsc = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_backward(prec, tc, dev(dout, dt), d_qkv, out, lse, dqkv, Dsc, B, T, C, NH)
    G.gpt2_device_status()
    tol = 2e-2 if bf16 else 1e-5
    assert rel_to_max(host(out), ref_out) < tol
    got = host(dqkv).reshape(B, T, 3, C)
    ref = ref_dqkv.reshape(B, T, 3, C)
    for part in range(3):
        assert rel_to_max(got[:, :, part], ref[:, :, part]) < (3e-2 if bf16 else 1e-5), part


@pytest.mark.parametrize("T", [1024, 300])
def test_attention_growing_scores_match_oracle(T):
    """Scores that climb by ~15 (log2 units) per 128-key block, so the online
    softmax must move its running maximum many times along a row."""
    import torch
    B, C, NH = 1, 128, 2
    q = np.full((B, T, C), 0.5, np.float32)
    ramp = (np.arange(T, dtype=np.float32) / T * 20.0)[None, :, None]
    k = ramp + inputs.normal(11, 1, B * T * C, 0.3).reshape(B, T, C).astype(np.float32)
    v = inputs.normal(11, 2, B * T * C).reshape(B, T, C).astype(np.float32)
    qkv = inputs.round_to_bf16(np.concatenate([q, k, v], axis=2).reshape(-1))
    dout = inputs.round_to_bf16(inputs.normal(11, 3, B * T * C, 0.1).astype(np.float32))
    ref_out, att = oracle.attention_forward(qkv, B, T, C, NH)
    ref_dqkv = oracle.attention_backward(dout, qkv, att, B, T, C, NH)
    d_qkv = dev(qkv, "bf16")
    out = empty((B * T * C,), "bf16")
    lse = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_forward(G.GPT2_BF16, 1, d_qkv, out, lse, B, T, C, NH)
    dqkv = empty((B * T * 3 * C,), "bf16")
    Dsc = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_backward(G.GPT2_BF16, 1, dev(dout, "bf16"), d_qkv, out, lse, dqkv, Dsc,
                              B, T, C, NH)
    G.gpt2_device_status()
    assert rel_to_max(host(out), ref_out) < 2e-2
    # log-sum-exp of the scaled causal scores, per (head, query)
    x = qkv.astype(np.float64).reshape(B, T, 3, NH, C // NH)
    s = np.einsum("tnd,snd->nts", x[0, :, 0], x[0, :, 1]) / np.sqrt(C // NH)
    s = np.where(np.tril(np.ones((T, T), bool))[None], s, -np.inf)
    mx = s.max(-1, keepdims=True)
    ref_lse = (mx + np.log(np.exp(s - mx).sum(-1, keepdims=True)))[..., 0]
    np.testing.assert_allclose(host(lse).reshape(NH, T), ref_lse, atol=2e-3, rtol=1e-4)
    got = host(dqkv).reshape(B, T, 3, C)
    ref = ref_dqkv.reshape(B, T, 3, C)
    # dK and dV as in the other cases. dQ sums dS_ij K_j over keys whose common
    # offset (the ramp, up to 20) cancels exactly because each row of dS sums to
    # zero; dS is rounded to bf16 first, so what survives is ~2^-9 of the
    # offset per term and the bound is looser.
    assert rel_to_max(got[:, :, 1], ref[:, :, 1]) < 3e-2
    assert rel_to_max(got[:, :, 2], ref[:, :, 2]) < 3e-2
    assert rel_to_max(got[:, :, 0], ref[:, :, 0]) < 1.5e-1


@pytest.mark.parametrize("B,T,C,NH", [(10, 1024, 256, 4), (40, 300, 128, 2)])
def test_attention_forward_many_items_per_cta(B, T, C, NH):
    """More (b, h, 256-query) work items than SMs, so the persistent forward
    runs several items per CTA (its Q buffers, K/V ring and TMEM regions are
    reused across items); T=300 also has items whose second query tile is
    empty. Output against the oracle, LSE against its definition."""
    import torch
    qkv = inputs.round_to_bf16(inputs.normal(40 + T, 1, B * T * 3 * C).astype(np.float32))
    ref_out = np.concatenate([
        oracle.attention_forward(qkv.reshape(B, -1)[b], 1, T, C, NH)[0] for b in range(B)])
    out = empty((B * T * C,), "bf16")
    lse = torch.zeros(B * NH * T, dtype=torch.float32, device="cuda")
    G.gpt2_attention_forward(G.GPT2_BF16, 1, dev(qkv, "bf16"), out, lse, B, T, C, NH)
    G.gpt2_device_status()
    assert rel_to_max(host(out), ref_out) < 2e-2
    x = qkv.astype(np.float64).reshape(B, T, 3, NH, C // NH)
    mask = np.tril(np.ones((T, T), bool))
    got_lse = host(lse).reshape(B, NH, T)
    for b in range(B):
        s = np.einsum("tnd,snd->nts", x[b, :, 0], x[b, :, 1]) / np.sqrt(C // NH)
        s = np.where(mask[None], s, -np.inf)
        mx = s.max(-1, keepdims=True)
        ref_lse = (mx + np.log(np.exp(s - mx).sum(-1, keepdims=True)))[..., 0]
        np.testing.assert_allclose(got_lse[b], ref_lse, atol=2e-3, rtol=1e-4)


def test_fused_op_small_shapes_match_oracle():
    import torch
    # (1024 x 9728 takes the 256-column tiles, the others the 224-column ones)
    for (M, K, N) in [(130, 72, 264), (256, 512, 1000), (1, 4, 4), (1024, 64, 9728)]:
        x, W, b = inputs.fused_op_inputs(M, K, N, seed=3)
        ref = oracle.fused_linear_bias_gelu_softmax(x, W, b)
        out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
        G.fused_linear_bias_gelu_softmax(dev(x), dev(W), dev(b), out, M, K, N)
        G.gpt2_device_status()
        y = host(out)
        np.testing.assert_allclose(y.sum(1), 1.0, atol=1e-5)
        assert max_rel_floor(y, ref, 0.0) < 1e-3, (M, K, N, max_rel_floor(y, ref, 0.0))


@pytest.mark.parametrize("N,C,dt", [(1000, 768, "bf16"), (37, 64, "f32"), (8192, 768, "bf16"),
                                    (300, 1024, "bf16"), (129, 1024, "f32"), (515, 640, "bf16"),
                                    (700, 512, "bf16"), (9, 256, "bf16"), (4096, 1024, "bf16")])
def test_layernorm_forward_backward_match_oracle(N, C, dt):
    import torch
    bf16 = dt == "bf16"
    x = inputs.normal(N + C, 1, N * C, 2.0).reshape(N, C).astype(np.float32) + 0.5
    w = (1.0 + inputs.normal(N + C, 2, C, 0.1)).astype(np.float32)
    b = inputs.normal(N + C, 3, C, 0.1).astype(np.float32)
    dy = inputs.normal(N + C, 4, N * C, 0.01).reshape(N, C).astype(np.float32)
    d0 = inputs.normal(N + C, 5, N * C, 0.01).reshape(N, C).astype(np.float32)
    if bf16:
        x, w, b, dy, d0 = (inputs.round_to_bf16(a) for a in (x, w, b, dy, d0))
    ref, mean, rstd = oracle.layernorm_forward(x, w, b)
    prec = G.GPT2_BF16 if bf16 else G.GPT2_FP32
    out = empty((N, C), dt)
    dmean = torch.zeros(N, device="cuda")
    drstd = torch.zeros(N, device="cuda")
    dx = dev(x, dt)
    G.gpt2_layernorm_forward(prec, out, dmean, drstd, dx, dev(w, dt), dev(b, dt), N, C)
    tol = 1e-2 if bf16 else 1e-5
    assert rel_to_max(host(out), ref) < tol
    np.testing.assert_allclose(host(drstd), rstd, rtol=1e-4)
    # backward, accumulating into d0 and into nonzero dw, db
    dinp = d0.astype(np.float64).copy()
    dw = np.ones(C)
    db = np.ones(C)
    oracle.layernorm_backward(dinp, dw, db, dy, x, w, mean, rstd)
    g_dinp = dev(d0, dt)
    g_dw = dev(np.ones(C, dtype=np.float32), dt)
    g_db = dev(np.ones(C, dtype=np.float32), dt)
    scratch = torch.zeros(G.gpt2_layernorm_backward_scratch_floats(C), device="cuda")
    G.gpt2_layernorm_backward(prec, g_dinp, g_dw, g_db, dev(dy, dt), dx, dev(w, dt), dmean, drstd, N,
                              C, 1, scratch)
    G.gpt2_device_status()
    assert rel_to_max(host(g_dinp), dinp) < (2e-2 if bf16 else 1e-5)
    # dw, db = 1 + sums over rows: the bf16 result is rounded once near 1 (a
    # half ulp is 2^-8), on top of the sums' own relative error
    for got, want in ((host(g_dw), dw), (host(g_db), db)):
        err = np.max(np.abs(got - want))
        if bf16:
            assert err <= 2.0 ** -8 * np.max(np.abs(want)) + 2e-2 * np.max(np.abs(want - 1.0))
        else:
            assert rel_to_max(got - 1.0, want - 1.0) < 1e-5


def test_stand_alone_entry_points_reject_bad_arguments_with_a_message():
    """Degenerate and misaligned calls are refused on the host, before any
    launch, with the code the header documents and a description of this call
    in gpt2_last_error; a valid call afterwards still runs."""
    import torch
    f32 = lambda *s: torch.zeros(*s, device="cuda")  # noqa: E731
    x, W, b, out = f32(8, 8), f32(8, 8), f32(8), f32(8, 8)

    def refused(code, text, fn, *args, **kw):
        with pytest.raises(G.GPT2Error) as e:
            fn(*args, **kw)
        assert e.value.code == code, e.value
        assert text in G.gpt2_last_error(), G.gpt2_last_error()
        assert G.gpt2_last_status() == code

    for fused in (G.fused_linear_bias_gelu_softmax, G.fused_linear_bias_gelu_softmax_noalloc):
        name = fused.__name__
        refused(-8, name if fused is G.fused_linear_bias_gelu_softmax else "M, K, N", fused,
                x, W, b, out, 0, 8, 8)  # empty input
        refused(-8, "NULL", fused, None, W, b, out, 8, 8, 8)
        refused(-5, "align", fused, x, W, b, out, 8, 6, 8)  # K not a multiple of 4
        refused(-5, "align", fused, x[:, 1:], W, b, out, 8, 4, 4)  # x not 16-byte aligned
    A, B, D = (torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    refused(-8, "gpt2_gemm", G.gpt2_gemm, G.GPT2_BF16, 1, "store", A, 64, 1, B, 64, 1, D, 64,
            M=0, N=64, K=64)
    refused(-8, "gpt2_gemm", G.gpt2_gemm, G.GPT2_BF16, 1, "store", A, 64, 1, B, 64, 1, D, 64,
            M=64, N=64, K=0)
    refused(-5, "gpt2_gemm", G.gpt2_gemm, G.GPT2_BF16, 1, "store", A, 64, 1, B, 64, 1, D, 64,
            M=64, N=60, K=64)  # N not a multiple of 8 bf16 values
    refused(-1, "gpt2_gemm", G.gpt2_gemm, 7, 1, "store", A, 64, 1, B, 64, 1, D, 64,
            M=64, N=64, K=64)  # unknown dtype
    refused(-8, "gpt2_gemm", G.gpt2_gemm, G.GPT2_BF16, 1, "resid", A, 64, 1, B, 64, 1, D, 64,
            M=64, N=64, K=64)  # residual epilogue without its operand
    qkv = torch.zeros(2 * 16 * 3 * 96, dtype=torch.bfloat16, device="cuda")
    o = torch.zeros(2 * 16 * 96, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(2 * 16 * 2, device="cuda")
    refused(-8, "gpt2_attention_forward", G.gpt2_attention_forward, G.GPT2_BF16, 1, qkv, o, lse,
            2, 16, 96, 5)  # C not a multiple of NH
    refused(-1, "gpt2_attention_forward", G.gpt2_attention_forward, G.GPT2_BF16, 1, qkv, o, lse,
            2, 16, 96, 2)  # head size 48
    refused(-8, "gpt2_attention_forward", G.gpt2_attention_forward, G.GPT2_BF16, 1, qkv, o, lse,
            0, 16, 96, 3)  # empty batch
    ln_out, mean, rstd = f32(4, 16), f32(4), f32(4)
    refused(-8, "gpt2_layernorm_forward", G.gpt2_layernorm_forward, G.GPT2_FP32, ln_out, mean, rstd,
            ln_out, f32(16), f32(16), 4, 12)  # C not a multiple of 8
    refused(-8, "gpt2_layernorm_forward", G.gpt2_layernorm_forward, G.GPT2_FP32, ln_out, mean, rstd,
            ln_out, f32(16), f32(16), 0, 16)  # no rows
    # the library is still usable: a valid product runs and is exact on integers
    A.copy_(torch.eye(64, dtype=torch.bfloat16, device="cuda") * 2)
    B.copy_(torch.arange(64 * 64, device="cuda").reshape(64, 64).remainder(7).to(torch.bfloat16))
    G.gpt2_gemm(G.GPT2_BF16, 1, "store", A, 64, 1, B, 64, 1, D, 64, M=64, N=64, K=64)
    G.gpt2_device_status()
    assert torch.equal(D.float(), 2 * B.float().T)
