"""GPU parity of per-question temperature sampling against the CPU oracle.

Greedy tokens (temperature 0) are unique: they must equal the oracle's.  A sampled token k is
correct when its interval of the cumulative distribution holds the question's uniform u; the
kernel sums ~1.5e5 weights in fp32, so near a boundary (within 5e-5 of the float64 cumulative
distribution) either neighbour is accepted, and with a small vocabulary (boundaries far apart)
the tokens must equal the oracle's."""
import numpy as np
import pytest
import torch

import packed_question_isolated_gb300 as kev
import workloads as W
from oracle import kev_oracle as O

from kev_harness import dev, host

pytestmark = pytest.mark.gpu

TOL = 5e-5


def _run(logits_stored, dtype, temperature, uniforms, active, sentinel=-7):
    n, vocab = logits_stored.shape
    tokens = torch.full((n,), sentinel, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kev.kev_sample(dev(logits_stored), n, vocab, dtype, torch.tensor(temperature, dtype=torch.float32).cuda(),
                   torch.tensor(uniforms, dtype=torch.float32).cuda(), torch.tensor(active, dtype=torch.uint8).cuda(),
                   tokens, st)
    return kev.kev_read_status(st), host(tokens)


def _assert_valid(tokens, logits64, temperature, uniforms, active, what):
    for i, tok in enumerate(tokens):
        if not active[i]:
            continue
        if temperature[i] == 0:
            assert tok == int(np.argmax(logits64[i])), f"{what}: question {i} greedy"
            continue
        cdf = np.cumsum(O.sample_probs(logits64[i], temperature[i]))
        lo = cdf[tok - 1] if tok > 0 else 0.0
        u = float(np.float32(uniforms[i]))
        assert lo - TOL <= u < cdf[tok] + TOL, f"{what}: question {i} token {tok}: u {u} outside [{lo}, {cdf[tok]})"


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_sample_large_vocab_is_valid(dtype):
    """64 questions over a 151,936-token vocabulary (the Qwen3 one), logits N(0, 2^2), temperatures
    0 (greedy), 0.3, 0.7, 1.0 and 1.5, a quarter of the questions dropped."""
    rng = np.random.default_rng(40)
    n, vocab = 64, 151936
    x = rng.standard_normal((n, vocab), dtype=np.float32) * 2
    x[3, [10, 99000]] = 30.0  # a tie at the maximum: greedy takes the lower index
    stored = W.f32_to_bf16_bits(x) if dtype == "bf16" else x
    logits64 = W.to_float64(stored, dtype)
    temperature = np.array([0.0, 0.3, 0.7, 1.0, 1.5, 0.0, 1.0, 0.7] * 8, np.float32)
    uniforms = rng.random(n).astype(np.float32)
    active = (rng.random(n) < 0.75).astype(np.uint8)
    active[3] = 1
    status, tokens = _run(stored, dtype, temperature, uniforms, active)
    assert status == 0
    assert tokens[3] == 10
    assert (tokens[active == 0] == -7).all()  # dropped questions: untouched
    _assert_valid(tokens, logits64, temperature.astype(np.float64), uniforms, active, f"{dtype} large vocab")
    ref = O.sample_tokens(logits64, temperature.astype(np.float64), uniforms.astype(np.float64), active)
    live = active.astype(bool)
    # tokens that differ from the oracle's lie next to a boundary: a few indices away at most
    assert np.abs(tokens[live] - ref[live]).max() <= 64


def test_sample_small_vocab_matches_the_oracle_and_the_probabilities():
    """4096 questions with the same 8 logits and uniforms on a grid: the tokens equal the oracle's,
    and their frequencies are the softmax probabilities."""
    n = 4096
    lg = np.array([0.5, -1.0, 2.0, 0.0, 1.5, -0.5, 0.25, 1.0], np.float32)
    logits = np.tile(lg, (n, 1))
    uniforms = ((np.arange(n) + 0.5) / n).astype(np.float32)
    for T in (0.5, 1.0, 2.5):
        temperature = np.full(n, T, np.float32)
        status, tokens = _run(logits, "fp32", temperature, uniforms, np.ones(n, np.uint8))
        assert status == 0
        ref = O.sample_tokens(logits.astype(np.float64), temperature.astype(np.float64),
                              uniforms.astype(np.float64))
        assert (tokens != ref).sum() <= 2  # only a uniform within rounding of a boundary may differ
        freq = np.bincount(tokens, minlength=8) / n
        p = O.sample_probs(lg, T)
        np.testing.assert_allclose(freq, p, atol=2.0 / n + 1e-6)


def test_invalid_temperature_or_uniform_writes_no_token():
    rng = np.random.default_rng(41)
    x = rng.standard_normal((4, 64), dtype=np.float32)
    for temperature, uniforms, active in (([1.0, -0.5, 1.0, 1.0], [0.1, 0.2, 0.3, 0.4], [1, 1, 1, 1]),
                                          ([1.0, 1.0, np.inf, 1.0], [0.1, 0.2, 0.3, 0.4], [1, 1, 1, 1]),
                                          ([1.0, 1.0, 1.0, 1.0], [0.1, 1.0, 0.3, 0.4], [1, 1, 1, 1])):
        assert O.validate_sampling(temperature, uniforms, active) == O.SAMPLING
        status, tokens = _run(x, "fp32", np.array(temperature, np.float32), np.array(uniforms, np.float32),
                              np.array(active, np.uint8))
        assert status == kev.binding.KEV_ERR_SAMPLING
        assert (tokens == -7).all()
    # the same bad values on a dropped question are fine
    status, tokens = _run(x, "fp32", np.array([1.0, -0.5, 1.0, 1.0], np.float32),
                          np.array([0.1, 0.2, 0.3, 0.4], np.float32), np.array([1, 0, 1, 1], np.uint8))
    assert status == 0 and tokens[1] == -7 and (tokens[[0, 2, 3]] >= 0).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_sample_mass_in_later_segments(dtype):
    """A 32,000-token vocabulary (the row split over two CTAs) and the Qwen3 one (eight): the
    probability mass sits in one later part of the row per question (logits raised over a window),
    uniforms on a grid up to just below 1, so the token comes from every part of the row and from
    both ends of the cumulative distribution."""
    rng = np.random.default_rng(42)
    for vocab in (32000, 151936):
        n = 48
        x = rng.standard_normal((n, vocab), dtype=np.float32)
        for i in range(n):
            w0 = int(rng.integers(0, vocab - 4096))
            x[i, w0:w0 + 4096] += 6.0
        stored = W.f32_to_bf16_bits(x) if dtype == "bf16" else x
        logits64 = W.to_float64(stored, dtype)
        temperature = np.array([0.5, 1.0, 1.5, 0.0] * (n // 4), np.float32)
        uniforms = np.concatenate([(np.arange(n - 2) + 0.5) / (n - 2), [0.0, 0.99999994]]).astype(np.float32)
        active = np.ones(n, np.uint8)
        status, tokens = _run(stored, dtype, temperature, uniforms, active)
        assert status == 0
        _assert_valid(tokens, logits64, temperature.astype(np.float64), uniforms, active, f"{dtype} vocab {vocab}")
