"""The bounded in-kernel waits: with the wait limit shortened to 2 us, a large
tensor-core GEMM's waits run out; the kernel drains its in-flight copies and
MMAs, frees its tensor memory and returns, and the host sees
GPT2_ERR_DEVICE_TIMEOUT. With the default limit restored the next call
succeeds and is correct. (The shape has three 128-row blocks, so the GEMM runs
single-CTA MMAs: every copy it issues completes on its own barriers, which its
drain waits for.)"""
import numpy as np
import pytest

from transformer_lm_gb300 import gpt2 as G
from transformer_lm_gb300 import inputs
from tests.gpu_util import dev, empty, host, rel_to_max

pytestmark = pytest.mark.gpu


def test_expired_wait_is_reported_and_the_next_call_succeeds():
    M, N, K = 384, 8192, 8192
    A = inputs.round_to_bf16(inputs.normal(3, 1, M * K).astype(np.float32)).reshape(M, K)
    B = inputs.round_to_bf16(inputs.normal(3, 2, N * K, 0.02).astype(np.float32)).reshape(N, K)
    dA, dB = dev(A, "bf16"), dev(B, "bf16")
    D = empty((M, N), "bf16")
    G.gpt2_device_status()  # start clean
    try:
        G.gpt2_set_wait_limit(2000)
        G.gpt2_gemm(G.GPT2_BF16, 1, "store", dA, K, 1, dB, K, 1, D, N, M=M, N=N, K=K)
        with pytest.raises(G.GPT2Error) as e:
            G.gpt2_device_status()
        assert e.value.code == -9
    finally:
        G.gpt2_set_wait_limit(0)
    G.gpt2_gemm(G.GPT2_BF16, 1, "store", dA, K, 1, dB, K, 1, D, N, M=M, N=N, K=K)
    G.gpt2_device_status()
    rows = np.arange(0, M, 37)
    ref = A[rows].astype(np.float64) @ B.astype(np.float64).T
    assert rel_to_max(host(D)[rows], ref) < 8e-3
