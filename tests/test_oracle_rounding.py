"""Pins for the oracle's random numbers, stochastic rounding, AdamW without
master weights and softmax sampling (llm.c "train_gpt2.cu": random_u32 /
random_f32, SquirrelNoise5, stochastic_rounding, adamw_kernel3, sample_softmax).

Each test ties the oracle to something other than itself: torch's bf16
conversion, exhaustive enumeration of the rounding thresholds (which fixes the
probability of rounding up exactly), the float64 AdamW (pinned against
torch.optim.AdamW elsewhere), numpy's cumulative sum and search, and the
statistics any good hash or generator must show. The pages print no test
vectors for SquirrelNoise5 or xorshift*, so those two are pinned by their
statistics and by the GPU side, which implements them separately.
"""
import numpy as np
import torch

import oracle
from transformer_lm_gb300 import inputs


def _f32(bits):
    return np.array([bits], dtype=np.uint32).view(np.float32)[0]


def _bf16_value(bits16):
    return float(np.array([int(bits16) << 16], dtype=np.uint32).view(np.float32)[0])


def test_bf16_round_to_nearest_even_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 4000),
        # exact halfway cases between two bf16 values (ties to even both ways)
        np.array([0x3F808000, 0x3F818000, 0xBF808000, 0x00008000, 0x7F7F8000], dtype=np.uint32).view(np.float32),
        np.array([0.0, -0.0, np.inf, -np.inf, 1e-40, -1e-40], dtype=np.float32),
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in x], dtype=np.uint16)
    assert np.array_equal(got, ref)


def test_stochastic_rounding_over_all_thresholds_is_exact_and_unbiased():
    """Over all 65536 thresholds, a float rounds up exactly (low 16 bits) times
    and down otherwise; the mean of the results is the float itself."""
    for bits in (0x3F812345, 0x3F81FFFF, 0x3F810001, 0xC2ABCDEF, 0x3C000001, 0x3F7FFFFF, 0x00012345):
        x = float(_f32(bits))
        low = bits & 0xFFFF
        down = bits >> 16
        up = down + 1
        res = np.array([oracle.stochastic_round_bf16(x, r) for r in range(65536)])
        assert set(np.unique(res)) <= {down, up}
        assert int(np.sum(res == up)) == low
        mean = (np.sum(res == down) * _bf16_value(down) + np.sum(res == up) * _bf16_value(up)) / 65536.0
        assert mean == x, (hex(bits), mean, x)
        # only the low 16 bits of the random word are used
        assert all(oracle.stochastic_round_bf16(x, r) == oracle.stochastic_round_bf16(x, r | 0xABCD0000)
                   for r in range(0, 65536, 997))


def test_stochastic_rounding_leaves_bf16_values_unchanged():
    for bits16 in (0x3F80, 0xBF80, 0x4049, 0x0001, 0x7F7F, 0x0000):
        x = _bf16_value(bits16)
        assert all(oracle.stochastic_round_bf16(x, r) == bits16 for r in range(0, 65536, 331))


def test_squirrel_noise_bits_are_balanced_and_seed_dependent():
    n = 1 << 14
    out = np.array([oracle.squirrel_noise5(i, 12345) for i in range(n)], dtype=np.uint64)
    bits = (out[:, None] >> np.arange(32, dtype=np.uint64)) & np.uint64(1)
    freq = bits.mean(axis=0)
    assert np.all(np.abs(freq - 0.5) < 5 * 0.5 / np.sqrt(n)), freq
    # another seed: about half the bits differ, position by position
    out2 = np.array([oracle.squirrel_noise5(i, 12346) for i in range(n)], dtype=np.uint64)
    flips = np.array([bin(int(a ^ b)).count("1") for a, b in zip(out, out2)])
    assert abs(flips.mean() - 16.0) < 0.2
    # neighbouring positions are uncorrelated
    u = out.astype(np.float64) / 2.0 ** 32
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.05
    # the 2-D form at y = 0 is the 1-D hash
    assert all(oracle.noise_2d(i, 0, 7) == oracle.squirrel_noise5(i, 7) for i in range(100))


def test_xorshift_star_uniforms():
    r = oracle.Rng(1337)
    u = np.array([r.f32() for _ in range(20000)])
    assert np.all((u >= 0) & (u < 1))
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))  # 24-bit resolution
    # Kolmogorov-Smirnov distance to U(0,1)
    s = np.sort(u)
    ks = np.max(np.abs(s - np.arange(1, s.size + 1) / s.size))
    assert ks < 1.63 / np.sqrt(s.size)
    assert abs(np.corrcoef(u[:-1], u[1:])[0, 1]) < 0.05
    # the same state gives the same stream
    a, b = oracle.Rng(42), oracle.Rng(42)
    assert [a.u32() for _ in range(5)] == [b.u32() for _ in range(5)]


def _sr_case(n, seed):
    p = inputs.round_to_bf16(inputs.normal(seed, 1, n, 0.02)).astype(np.float32)
    g = inputs.round_to_bf16(inputs.normal(seed, 2, n, 1e-3)
                             * np.exp(inputs.normal(seed, 3, n, 1.0))).astype(np.float32)
    pb = (p.view(np.uint32) >> 16).astype(np.uint16)
    gb = (g.view(np.uint32) >> 16).astype(np.uint16)
    return p, g, pb, gb


def test_adamw_bf16_sr_rounds_the_float64_update_to_a_neighbour():
    n = 4096
    p, g, pb, gb = _sr_case(n, 3)
    m32, v32 = np.zeros(n, np.float32), np.zeros(n, np.float32)
    p64, m64, v64 = p.astype(np.float64), np.zeros(n), np.zeros(n)
    bits = pb.copy()
    rng = oracle.Rng(13371337)
    for t in (1, 2, 3):
        # the float64 update from the same (rounded) starting point
        p64 = np.array([_bf16_value(b) for b in bits])
        oracle.adamw(p64, g.astype(np.float64), m64, v64, 1e-3, 0.9, 0.95, 1e-8, 0.1, t)
        oracle.adamw_bf16_sr(bits, gb, m32, v32, 1e-3, 0.9, 0.95, 1e-8, 0.1, t, rng.u32())
        np.testing.assert_allclose(m32, m64, rtol=1e-5, atol=1e-12)
        np.testing.assert_allclose(v32, v64, rtol=1e-5, atol=1e-16)
        got = np.array([_bf16_value(b) for b in bits])
        # each result is one of the two bf16 values around the float64 update
        # (up to the float32 rounding of the update itself)
        below = np.array([_bracket(x)[0] for x in p64])
        above = np.array([_bracket(x)[1] for x in p64])
        tol = 4 * np.abs(p64) * 2.0 ** -24
        ok = ((got >= below - tol) & (got <= above + tol))
        assert ok.all(), np.flatnonzero(~ok)[:5]


def _bracket(x):
    """The two bf16 values around x (equal when x is one)."""
    b = int(np.array([x], dtype=np.float32).view(np.uint32)[0])
    trunc = _bf16_value(b >> 16)
    nxt = _bf16_value((b >> 16) + 1)
    return (min(trunc, nxt), max(trunc, nxt)) if trunc != x else (trunc, trunc)


def test_adamw_bf16_sr_is_unbiased_over_seeds():
    """Averaged over many step seeds, the stochastically rounded parameter
    equals the float update (its expectation), where round-to-nearest would
    keep a bias of up to half a bf16 ulp."""
    n, reps = 256, 1500
    p, g, pb, gb = _sr_case(n, 5)
    acc = np.zeros(n)
    rng = oracle.Rng(99)
    for _ in range(reps):
        bits = pb.copy()
        m32, v32 = np.zeros(n, np.float32), np.zeros(n, np.float32)
        oracle.adamw_bf16_sr(bits, gb, m32, v32, 1e-3, 0.9, 0.95, 1e-8, 0.1, 1, rng.u32())
        acc += np.array([_bf16_value(b) for b in bits])
    mean = acc / reps
    p64 = p.astype(np.float64)
    oracle.adamw(p64, g.astype(np.float64), np.zeros(n), np.zeros(n), 1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    ulp = np.array([_bracket(x)[1] - _bracket(x)[0] for x in p64])
    # per element: within 5 standard errors of a Bernoulli over one ulp
    assert np.all(np.abs(mean - p64) <= 5 * 0.5 * ulp / np.sqrt(reps) + 4 * np.abs(p64) * 2.0 ** -24)
    # and the mean error over elements is far below round-to-nearest's
    assert abs(np.mean((mean - p64) / np.maximum(ulp, 1e-30))) < 0.02


def test_sample_softmax_against_numpy_cdf():
    rng = np.random.default_rng(3)
    for n in (1, 7, 1000):
        logits = rng.standard_normal(n) * 3
        p = np.exp(logits - logits.max())
        cdf = np.cumsum(p / p.sum())
        for coin in rng.random(200):
            i = oracle.sample_softmax(logits, coin)
            j = min(int(np.searchsorted(cdf, coin, side="right")), n - 1)
            near = np.min(np.abs(cdf - coin)) < 1e-12
            assert i == j or near, (n, coin, i, j)
    # special cases: a dominant logit, equal logits, coin 0
    lg = np.zeros(50)
    lg[17] = 100.0
    assert all(oracle.sample_softmax(lg, c) == 17 for c in (1e-9, 0.3, 0.999))
    assert oracle.sample_softmax(lg, 0.0) == 0  # the first index whose cdf exceeds 0
    eq = np.zeros(64)
    assert all(oracle.sample_softmax(eq, c) == int(np.floor(c * 64)) for c in (0.0, 0.01, 0.5, 0.99))
