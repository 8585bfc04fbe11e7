"""The allocation-free fused Linear+bias+GELU+softmax entry point.

It is for callers that cannot let the library allocate device memory: its
scratch is a static device array, so it must give the same output as the
allocating entry point, call after call (the shared array keeps the previous
call's contents), and refuse sizes beyond that array with a clear error.
This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import numpy as np
import pytest

from transformer_lm_gb300 import gpt2 as G
from transformer_lm_gb300 import inputs

pytestmark = pytest.mark.gpu

TOL = 2e-2  # single-pass TF32 here against the split-bf16 allocating entry (max relative difference)


def _run(fn, M, K, N, seed):
    import torch
    x, W, b = inputs.fused_op_inputs(M, K, N, seed=seed)
    out = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    fn(torch.from_numpy(x).cuda(), torch.from_numpy(W).cuda(), torch.from_numpy(b).cuda(), out,
       M, K, N)
    G.gpt2_device_status()
    return out.cpu().numpy().astype(np.float64)


def test_noalloc_matches_allocating_entry_point_on_two_calls_in_a_row():
    # two different shapes back to back: the second call reuses the static
    # scratch the first one left behind
    for (M, K, N, seed) in [(300, 512, 1000, 5), (128, 256, 512, 6)]:
        ref = _run(G.fused_linear_bias_gelu_softmax, M, K, N, seed)
        got = _run(G.fused_linear_bias_gelu_softmax_noalloc, M, K, N, seed)
        rel = np.max(np.abs(got - ref) / np.abs(ref))
        assert rel <= TOL, (M, K, N, rel)
        np.testing.assert_allclose(got.sum(1), 1.0, atol=1e-5)


def test_noalloc_rejects_sizes_beyond_its_static_scratch():
    import torch
    M, K, N = 1025, 4, 32768  # 1025 * 128 tiles > 131072 partials
    x = torch.zeros((M, K), device="cuda")
    W = torch.zeros((N, K), device="cuda")
    b = torch.zeros(N, device="cuda")
    out = torch.zeros((M, N), device="cuda")
    with pytest.raises(G.GPT2Error) as e:
        G.fused_linear_bias_gelu_softmax_noalloc(x, W, b, out, M, K, N)
    assert e.value.code == -8
    assert "static scratch" in str(e.value)
