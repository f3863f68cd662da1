"""Randomised pins of the oracle: on random small shapes, prefix ladders, scales and biases the
float64 oracle equals torch's cross_entropy / logsigmoid with autograd, prefix by prefix
(the loss definitions of "Scaling-Up Contrastive Learning over NVLink Multicast", section
"One Set or Two"; Matryoshka prefixes each normalised on their own)."""
import os

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings  # noqa: E402
from hypothesis import strategies as st  # noqa: E402

import oracle  # noqa: E402
from test_oracle_pins import _bits, _wide, torch_reference  # noqa: E402

EPS = np.finfo(np.float64).eps


@st.composite
def problems(draw):
    kind = draw(st.sampled_from(["clip", "siglip", "rows"]))
    Na = draw(st.integers(1, 10))
    Nb = Na if kind == "clip" else draw(st.integers(Na, Na + 6))
    D = draw(st.sampled_from([64, 128, 192]))
    ends = draw(st.lists(st.sampled_from(range(16, D + 1, 16)), min_size=1, max_size=5, unique=True))
    prefixes = tuple(sorted(ends))
    if kind == "siglip":
        scale = draw(st.floats(0.5, 20.0))
        bias = draw(st.floats(-15.0, 5.0))
    else:
        scale = draw(st.floats(0.5, 40.0))
        bias = 0.0
    noise = draw(st.floats(0.05, 2.0))
    seed = draw(st.integers(0, 2**31 - 1))
    return kind, Na, Nb, D, prefixes, scale, bias, noise, seed


# ORACLE_PROPERTY_EXAMPLES raises the number of drawn problems for a longer run
@settings(max_examples=int(os.environ.get("ORACLE_PROPERTY_EXAMPLES", "60")), deadline=None)
@given(problems())
def test_oracle_matches_torch_on_random_problems(prob):
    kind, Na, Nb, D, prefixes, scale, bias, noise, seed = prob
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((Na, D))
    b = np.concatenate([a, rng.standard_normal((Nb - Na, D))])[:Nb] + noise * rng.standard_normal((Nb, D))
    A, B = _bits(a), _bits(b)
    weights = rng.uniform(0.5, 2.0, len(prefixes))
    got = oracle.fwd_bwd(kind, A, B, prefixes, scale, bias, weights)
    L, gA, gB = torch_reference(kind, _wide(A), _wide(B), prefixes, scale, bias, weights)
    # both sides form a log-sum-exp less the positive logit around s = scale: below a few
    # ulp(scale) the difference is rounding, so that is the absolute floor
    floor = 64 * EPS * scale
    np.testing.assert_allclose(got["loss"], L, rtol=1e-11, atol=floor)
    # a gradient entry is (softmax or sigmoid, less the label) * scale * rho * O(1): near
    # saturation that difference cancels, so its rounding floor is a few ulp of scale * rho
    xa, xb = _wide(A), _wide(B)
    rho = max(1.0 / np.linalg.norm(x[:, :p], axis=1).min() for x in (xa, xb) for p in prefixes)
    gfloor = 64 * EPS * scale * rho * max(weights)
    np.testing.assert_allclose(got["dA"], gA, rtol=1e-9, atol=gfloor)
    np.testing.assert_allclose(got["dB"], gB, rtol=1e-9, atol=gfloor)
