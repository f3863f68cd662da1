"""Pins for the float64 oracle: checks against things other than the oracle itself.

Each pin ties the oracle to something the pages or mathematics fix:
  * closed forms (identical embeddings give InfoNCE = ln N and SigLIP = N ln 2 with
    zero gradients; one-hot orthogonal rows give ln(1 + (N-1) e^-tau));
  * library routines: torch's cross_entropy / logsigmoid for each prefix's loss and
    torch autograd for the gradients (an independent derivation of the chain rule);
  * brute-force central finite differences on tiny float64 inputs;
  * invariants: A<->B swap symmetry, ROWS(A,B) + ROWS(B,A) = 2 CLIP(A,B), per-row
    scale invariance and its Euler identity, permutation equivariance.
A dropped term, a wrong sign or index, or a transposed operand in the oracle fails at
least one of these (see the planted-mistake tests at the end).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from contrastive_embedding_loss_gb300 import synth


def _bits(x):
    return synth.round_to_bf16_bits(np.asarray(x, np.float64))


def _wide(bits):
    return synth.bf16_bits_to_float(bits).astype(np.float64)


def torch_reference(kind, A, B, prefixes, scale, bias, weights):
    """Per-prefix losses and gradients from torch library routines + autograd (float64)."""
    At = torch.tensor(A, dtype=torch.float64, requires_grad=True)
    Bt = torch.tensor(B, dtype=torch.float64, requires_grad=True)
    Na, Nb = At.shape[0], Bt.shape[0]
    losses, total = [], 0.0
    for p, w in zip(prefixes, weights):
        a = F.normalize(At[:, :p], dim=1, eps=1e-30)
        b = F.normalize(Bt[:, :p], dim=1, eps=1e-30)
        cos = a @ b.T
        if kind == "clip":
            s = scale * cos
            t = torch.arange(Na)
            L = 0.5 * (F.cross_entropy(s, t) + F.cross_entropy(s.T, t))
        elif kind == "rows":
            L = F.cross_entropy(scale * cos, torch.arange(Na))
        else:
            x = scale * cos + bias
            z = 2.0 * torch.eye(Na, Nb, dtype=torch.float64) - 1.0
            L = -F.logsigmoid(z * x).sum() / Na
        losses.append(L.item())
        total = total + w * L
    total.backward()
    return np.array(losses), At.grad.numpy(), Bt.grad.numpy()


CASES = [
    ("clip", 12, 12, 192, (64, 128, 192), 1 / 0.07, 0.0),
    ("siglip", 10, 10, 128, (32, 64, 128), 10.0, -10.0),
    ("rows", 6, 15, 128, (64, 128), 1 / 0.05, 0.0),
    ("clip", 9, 9, 128, (128,), 3.0, 0.0),
    ("siglip", 6, 10, 128, (64, 128), 4.0, -2.0),   # columns past Na: extra negatives only
]


@pytest.mark.parametrize("kind,Na,Nb,D,prefixes,scale,bias", CASES)
def test_matches_torch_library_and_autograd(kind, Na, Nb, D, prefixes, scale, bias):
    rng = np.random.default_rng(7)
    a = rng.standard_normal((Na, D))
    b = np.concatenate([a, rng.standard_normal((Nb - Na, D))])[:Nb] + 0.8 * rng.standard_normal((Nb, D))
    A, B = _bits(a), _bits(b)
    weights = rng.uniform(0.5, 2.0, len(prefixes))
    got = oracle.fwd_bwd(kind, A, B, prefixes, scale, bias, weights)
    L, gA, gB = torch_reference(kind, _wide(A), _wide(B), prefixes, scale, bias, weights)
    np.testing.assert_allclose(got["loss"], L, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(got["dA"], gA, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(got["dB"], gB, rtol=1e-10, atol=1e-13)
    if kind == "rows":
        assert np.all(got["col_terms"] == 0)
    np.testing.assert_allclose(got["row_terms"].mean(axis=1) if kind == "rows" else got["loss"],
                               got["loss"], rtol=1e-13)


def torch_scale_grads(kind, A, B, prefixes, scale, bias, weights):
    """d(sum_k w_k L_k)/d(scale) and /d(bias) by torch autograd (float64), the scale and bias
    as leaves of the graph built from torch's cross_entropy / logsigmoid."""
    s = torch.tensor(float(scale), dtype=torch.float64, requires_grad=True)
    b_ = torch.tensor(float(bias), dtype=torch.float64, requires_grad=True)
    At = torch.tensor(A, dtype=torch.float64)
    Bt = torch.tensor(B, dtype=torch.float64)
    Na, Nb = At.shape[0], Bt.shape[0]
    total = 0.0
    for p, w in zip(prefixes, weights):
        cos = F.normalize(At[:, :p], dim=1, eps=1e-30) @ F.normalize(Bt[:, :p], dim=1, eps=1e-30).T
        if kind == "clip":
            t = torch.arange(Na)
            L = 0.5 * (F.cross_entropy(s * cos, t) + F.cross_entropy((s * cos).T, t))
        elif kind == "rows":
            L = F.cross_entropy(s * cos, torch.arange(Na))
        else:
            z = 2.0 * torch.eye(Na, Nb, dtype=torch.float64) - 1.0
            L = -F.logsigmoid(z * (s * cos + b_)).sum() / Na
        total = total + w * L
    total.backward()
    return s.grad.item(), (b_.grad.item() if b_.grad is not None else 0.0)


@pytest.mark.parametrize("kind,Na,Nb,D,prefixes,scale,bias", CASES)
def test_scale_grads_match_autograd(kind, Na, Nb, D, prefixes, scale, bias):
    rng = np.random.default_rng(17)
    a = rng.standard_normal((Na, D))
    b = np.concatenate([a, rng.standard_normal((Nb - Na, D))])[:Nb] + 0.8 * rng.standard_normal((Nb, D))
    A, B = _bits(a), _bits(b)
    weights = rng.uniform(0.5, 2.0, len(prefixes))
    ds, db = oracle.scale_grads(kind, A, B, prefixes, scale, bias, weights)
    ts, tb = torch_scale_grads(kind, _wide(A), _wide(B), prefixes, scale, bias, weights)
    np.testing.assert_allclose(ds, ts, rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(db, tb, rtol=1e-10, atol=1e-13)
    if kind != "siglip":
        assert db == 0.0


@pytest.mark.parametrize("kind", ["clip", "siglip", "rows"])
def test_scale_grads_finite_differences(kind):
    """Central differences of the oracle's own weighted loss in the scale and the bias."""
    rng = np.random.default_rng(19)
    Na, Nb, D = 5, (7 if kind == "rows" else 5), 16
    prefixes = (8, 16)
    A = rng.standard_normal((Na, D))
    B = rng.standard_normal((Nb, D))
    B[:Na] += A
    scale, bias = (2.5, -1.5) if kind == "siglip" else (3.0, 0.0)
    w = np.array([0.7, 1.3])
    ds, db = oracle.scale_grads(kind, A, B, prefixes, scale, bias, w)

    def f(s_, b_):
        return float(np.dot(w, oracle.fwd_bwd(kind, A, B, prefixes, s_, b_, w, grads=False)["loss"]))

    h = 1e-6
    np.testing.assert_allclose(ds, (f(scale + h, bias) - f(scale - h, bias)) / (2 * h), rtol=1e-6, atol=1e-9)
    if kind == "siglip":
        np.testing.assert_allclose(db, (f(scale, bias + h) - f(scale, bias - h)) / (2 * h), rtol=1e-6, atol=1e-9)


def test_scale_grads_closed_forms():
    N, D = 6, 64
    pre = (32, 64)
    # identical rows: every cosine is 1; InfoNCE's expected cosine equals the positive's (0),
    # SigLIP at t = 10, b = -10 has x = 0 and sigmoid = 1/2 everywhere: 0.5 N - 1 per prefix
    v = np.random.default_rng(3).standard_normal(D)
    X = _bits(np.tile(v, (N, 1)))
    ds, db = oracle.scale_grads("clip", X, X, pre, 5.0, 0.0)
    assert abs(ds) < 1e-12 and db == 0.0
    ds, db = oracle.scale_grads("siglip", X, X, pre, 10.0, -10.0)
    np.testing.assert_allclose([ds, db], [len(pre) * (0.5 * N - 1)] * 2, rtol=1e-12)
    # one-hot orthogonal rows: cos = [i == j]
    E = _bits(np.eye(N, D))
    tau = 4.0
    ds, _ = oracle.scale_grads("clip", E, E, pre, tau, 0.0)
    np.testing.assert_allclose(ds, len(pre) * -(N - 1) / (math.exp(tau) + N - 1), rtol=1e-12)
    t, b = 3.0, -2.0
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))  # noqa: E731
    ds, db = oracle.scale_grads("siglip", E, E, pre, t, b)
    np.testing.assert_allclose(ds, len(pre) * (sig(t + b) - 1.0), rtol=1e-12)
    np.testing.assert_allclose(db, len(pre) * (sig(t + b) - 1.0 + (N - 1) * sig(b)), rtol=1e-12)


@pytest.mark.parametrize("kind", ["clip", "siglip", "rows"])
def test_finite_differences(kind):
    rng = np.random.default_rng(11)
    Na, Nb, D = 4, (6 if kind == "rows" else 4), 12
    prefixes = (4, 8, 12)
    A = rng.standard_normal((Na, D))
    B = rng.standard_normal((Nb, D))
    B[:Na] += A
    scale, bias = (2.5, -1.5) if kind == "siglip" else (3.0, 0.0)
    w = np.array([1.0, 0.5, 2.0])
    got = oracle.fwd_bwd(kind, A, B, prefixes, scale, bias, w)

    def f(A_, B_):
        return float(np.dot(w, oracle.fwd_bwd(kind, A_, B_, prefixes, scale, bias, w, grads=False)["loss"]))

    h = 1e-6
    for X, g in ((A, got["dA"]), (B, got["dB"])):
        num = np.zeros_like(X)
        for idx in np.ndindex(X.shape):
            x0 = X[idx]
            X[idx] = x0 + h
            fp = f(A, B)
            X[idx] = x0 - h
            fm = f(A, B)
            X[idx] = x0
            num[idx] = (fp - fm) / (2 * h)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8)


def test_identical_embeddings_closed_forms():
    rng = np.random.default_rng(3)
    v = rng.standard_normal(128)
    N = 8
    A = _bits(np.tile(v, (N, 1)))
    pre = (64, 128)
    clip = oracle.fwd_bwd("clip", A, A, pre, 1 / 0.07)
    np.testing.assert_allclose(clip["loss"], math.log(N), rtol=1e-13)
    assert np.abs(clip["dA"]).max() < 1e-12 and np.abs(clip["dB"]).max() < 1e-12
    sig = oracle.fwd_bwd("siglip", A, A, pre, 10.0, -10.0)
    np.testing.assert_allclose(sig["loss"], N * math.log(2.0), rtol=1e-13)
    assert np.abs(sig["dA"]).max() < 1e-12 and np.abs(sig["dB"]).max() < 1e-12
    K = _bits(np.tile(v, (9, 1)))
    rows = oracle.fwd_bwd("rows", A[:4], K, pre, 1 / 0.05)
    np.testing.assert_allclose(rows["loss"], math.log(9), rtol=1e-13)
    assert np.abs(rows["dA"]).max() < 1e-12 and np.abs(rows["dB"]).max() < 1e-12


def test_one_hot_orthogonal_closed_forms():
    N, D = 8, 128
    E = np.zeros((N, D))
    E[np.arange(N), np.arange(N) * 5] = 1.0
    A = _bits(E)
    tau = 1 / 0.07
    clip = oracle.fwd_bwd("clip", A, A, (64, 128), tau)
    # the oracle forms LSE - s_ii around s = tau, so allow a few ulp(tau) of absolute error
    np.testing.assert_allclose(clip["loss"], math.log1p((N - 1) * math.exp(-tau)), rtol=0, atol=1e-14)
    t, b = 10.0, -10.0
    sig = oracle.fwd_bwd("siglip", A, A, (64, 128), t, b)
    sp = lambda y: math.log1p(math.exp(y))  # noqa: E731
    np.testing.assert_allclose(sig["loss"], sp(-(t + b)) + (N - 1) * sp(b), rtol=1e-12)
    np.testing.assert_allclose(sig["loss"], math.log(2) + (N - 1) * 4.5398899216870535e-05, rtol=1e-9)


def _random_pair(N, D, seed, noise=1.0):
    return synth.paired(N, D, noise, seed)


def test_swap_symmetry():
    A, B = _random_pair(10, 128, 5)
    pre = (64, 128)
    for kind, s, b in (("clip", 1 / 0.07, 0.0), ("siglip", 10.0, -10.0)):
        r1 = oracle.fwd_bwd(kind, A, B, pre, s, b)
        r2 = oracle.fwd_bwd(kind, B, A, pre, s, b)
        np.testing.assert_allclose(r1["loss"], r2["loss"], rtol=1e-9, atol=1e-15)
        np.testing.assert_allclose(r1["dA"], r2["dB"], rtol=1e-10, atol=1e-14)
        np.testing.assert_allclose(r1["dB"], r2["dA"], rtol=1e-10, atol=1e-14)


def test_rows_identity():
    A, B = _random_pair(11, 128, 6)
    pre = (64, 128)
    tau = 1 / 0.07
    c = oracle.fwd_bwd("clip", A, B, pre, tau)
    r1 = oracle.fwd_bwd("rows", A, B, pre, tau)
    r2 = oracle.fwd_bwd("rows", B, A, pre, tau)
    np.testing.assert_allclose(r1["loss"] + r2["loss"], 2 * c["loss"], rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(r1["dA"] + r2["dB"], 2 * c["dA"], rtol=1e-9, atol=1e-14)


@pytest.mark.parametrize("kind", ["clip", "siglip", "rows"])
def test_scale_invariance_and_euler(kind):
    A, B = _random_pair(7, 128, 9)
    if kind == "rows":
        B = np.concatenate([B, _random_pair(5, 128, 10)[0]])
    pre = (64, 128)
    s, b = (10.0, -10.0) if kind == "siglip" else (1 / 0.07, 0.0)
    r = oracle.fwd_bwd(kind, A, B, pre, s, b)
    for X, G in ((A, r["dA"]), (B, r["dB"])):
        x = _wide(X)
        euler = np.abs((x * G).sum(axis=1))
        assert np.all(euler <= 1e-12 * (np.linalg.norm(x, axis=1) * np.linalg.norm(G, axis=1) + 1e-300))
    # scaling a row by 2 (exact in bf16) leaves the loss unchanged and halves its gradient
    A2 = _bits(2.0 * _wide(A))
    r2 = oracle.fwd_bwd(kind, A2, B, pre, s, b)
    np.testing.assert_allclose(r2["loss"], r["loss"], rtol=1e-9, atol=1e-15)
    np.testing.assert_allclose(r2["dA"], 0.5 * r["dA"], rtol=1e-9, atol=1e-15)


def test_permutation_equivariance():
    A, B = _random_pair(9, 128, 12)
    perm = np.random.default_rng(0).permutation(9)
    for kind, s, b in (("clip", 1 / 0.07, 0.0), ("siglip", 10.0, -10.0), ("rows", 1 / 0.05, 0.0)):
        r = oracle.fwd_bwd(kind, A, B, (64, 128), s, b)
        rp = oracle.fwd_bwd(kind, A[perm], B[perm], (64, 128), s, b)
        np.testing.assert_allclose(rp["loss"], r["loss"], rtol=1e-9, atol=1e-15)
        np.testing.assert_allclose(rp["dA"], r["dA"][perm], rtol=1e-10, atol=1e-15)
        np.testing.assert_allclose(rp["dB"], r["dB"][perm], rtol=1e-10, atol=1e-15)


def test_full_prefix_equals_unprefixed_cross_entropy():
    A, B = _random_pair(16, 256, 13)
    tau = 1 / 0.07
    r = oracle.fwd_bwd("clip", A, B, (64, 256), tau)
    a = F.normalize(torch.tensor(_wide(A)), dim=1)
    b = F.normalize(torch.tensor(_wide(B)), dim=1)
    s = tau * a @ b.T
    t = torch.arange(16)
    ce = 0.5 * (F.cross_entropy(s, t) + F.cross_entropy(s.T, t))
    np.testing.assert_allclose(r["loss"][-1], ce.item(), rtol=1e-12)


@pytest.mark.parametrize("kind", ["clip", "siglip", "rows"])
def test_sampled_row_functions_match_full(kind):
    Na, Nb = 12, (20 if kind == "rows" else 12)
    A, _ = _random_pair(Na, 128, 21)
    B, _ = _random_pair(Nb, 128, 22)
    B[:Na] = _bits(_wide(A) + 0.5 * _wide(B[:Na]))
    pre = (64, 128)
    s, b = (10.0, -10.0) if kind == "siglip" else (1 / 0.07, 0.0)
    w = np.array([0.7, 1.3])
    full = oracle.fwd_bwd(kind, A, B, pre, s, b, w)
    rows_a = np.array([0, 5, 11])
    rt = oracle.row_terms_sampled(kind, A, B, pre, s, b, rows_a)
    np.testing.assert_allclose(rt, full["row_terms"][:, rows_a], rtol=1e-12, atol=1e-14)
    lse_a, _ = oracle.row_stats(kind, A, B, pre, s, b, np.arange(Na))
    lse_b, _ = oracle.row_stats(kind, B, A, pre, s, b, np.arange(Nb))
    if kind == "clip":
        ct = oracle.row_terms_sampled(kind, B, A, pre, s, b, rows_a)
        np.testing.assert_allclose(ct, full["col_terms"][:, rows_a], rtol=1e-12, atol=1e-14)
    gA = oracle.grad_rows(kind, True, A, B, pre, s, b, rows_a, lse_a.T, lse_b.T, w)
    np.testing.assert_allclose(gA, full["dA"][rows_a], rtol=1e-10, atol=1e-15)
    rows_b = np.array([1, 7, Nb - 1])
    gB = oracle.grad_rows(kind, False, B, A, pre, s, b, rows_b, lse_b.T, lse_a.T, w)
    np.testing.assert_allclose(gB, full["dB"][rows_b], rtol=1e-10, atol=1e-15)


@pytest.mark.parametrize("kind", ["clip", "rows"])
def test_softmax_normalisers_match_the_row_loops_and_feed_full_gradients(kind):
    """The large-batch normalisers (one float64 matmul per prefix and row chunk) equal the C
    oracle's row loops; fed to grad_rows as lse_x / lse_y they give the full backward's rows."""
    Na, Nb = 70, (150 if kind == "rows" else 70)
    A, _ = _random_pair(Na, 128, 23)
    B, _ = _random_pair(Nb, 128, 24)
    B[:Na] = _bits(_wide(A) + 0.5 * _wide(B[:Na]))
    pre = (64, 128)
    s = 1 / 0.07
    lse_a, pos_a = oracle.softmax_normalisers(kind, A, B, pre, s, row_chunk=33)
    la, pa = oracle.row_stats(kind, A, B, pre, s, 0.0, np.arange(Na))
    np.testing.assert_allclose(lse_a, la.T, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(pos_a, pa.T, rtol=1e-13, atol=1e-13)
    lse_b, _ = oracle.softmax_normalisers(kind, B, A, pre, s, row_chunk=64)
    full = oracle.fwd_bwd(kind, A, B, pre, s, 0.0)
    rows = np.array([0, 33, Na - 1])
    gA = oracle.grad_rows(kind, True, A, B, pre, s, 0.0, rows, lse_a, lse_b)
    np.testing.assert_allclose(gA, full["dA"][rows], rtol=1e-10, atol=1e-15)
    cols = np.array([2, Na - 1, Nb - 1])
    gB = oracle.grad_rows(kind, False, B, A, pre, s, 0.0, cols, lse_b, lse_a)
    np.testing.assert_allclose(gB, full["dB"][cols], rtol=1e-10, atol=1e-15)
    # identical rows: every logit equals the scale, so lse = scale + ln N (the closed form)
    X = np.repeat(A[:1], 40, axis=0)
    lse, pos = oracle.softmax_normalisers(kind, X, X, pre, s)
    np.testing.assert_allclose(lse, s + math.log(40), rtol=1e-14)
    np.testing.assert_allclose(pos, s, rtol=1e-14)


def test_zero_norm_prefix_reading():
    """A row whose prefix is all zero scores cosine 0 there (inverse norm floored at 1e30)."""
    A, B = _random_pair(6, 128, 30)
    a = _wide(A)
    a[2, :64] = 0.0
    A = _bits_safe(a)
    r = oracle.fwd_bwd("clip", A, B, (64, 128), 1 / 0.07)
    assert np.all(np.isfinite(r["loss"])) and np.all(np.isfinite(r["dA"]))
    assert abs(r["row_terms"][0, 2] - math.log(6)) < 1e-12  # all six logits are 0


def _bits_safe(x):
    out = np.zeros(x.shape, np.uint16)
    nz = x != 0
    out[nz] = synth.round_to_bf16_bits(x[nz])
    return out


# ---- the input generator ----------------------------------------------------------

def test_bf16_rounding_matches_float32_bit_rounding():
    rng = np.random.default_rng(1)
    x = rng.standard_normal(100000).astype(np.float32)  # exactly representable inputs
    u = x.view(np.uint32).astype(np.uint64)
    ref = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)  # f32 -> bf16 RNE on the bits
    assert np.array_equal(synth.round_to_bf16_bits(x.astype(np.float64)), ref)
    # exact ties go to the even neighbour
    lo = synth.bf16_bits_to_float(np.array([0x3F80, 0x3F81], np.uint16)).astype(np.float64)
    assert synth.round_to_bf16_bits(np.array([(lo[0] + lo[1]) / 2]))[0] == 0x3F80
    lo = synth.bf16_bits_to_float(np.array([0x3F81, 0x3F82], np.uint16)).astype(np.float64)
    assert synth.round_to_bf16_bits(np.array([(lo[0] + lo[1]) / 2]))[0] == 0x3F82


def test_generators_are_seeded_and_chunk_invariant():
    A1, B1 = synth.paired(20000, 64, 1.0, 4)
    A2, B2 = synth.paired(20000, 64, 1.0, 4)
    assert np.array_equal(A1, A2) and np.array_equal(B1, B2)
    A3, _ = synth.paired(100, 64, 1.0, 4)
    assert np.array_equal(A3, A1[:100])
    Q, K = synth.queries_keys(50, 300, 64, 0.8, 4)
    assert Q.shape == (50, 64) and K.shape == (300, 64)
    c = np.corrcoef(_wide(Q[:, :]).ravel(), _wide(K[:50]).ravel())[0, 1]
    assert 0.7 < c < 0.85  # 1/sqrt(1 + 0.8^2) = 0.78
    Ah, Bh = synth.paired_hard(1000, 64, 1.0, 0.1, 0.05, 3)
    a = _wide(Ah)
    an = a / np.linalg.norm(a, axis=1, keepdims=True)
    near = (an @ an.T > 0.99).sum(axis=1) - 1
    assert 90 <= (near > 0).sum() <= 200  # ~100 duplicated rows, plus their sources


# ---- planted mistakes: each plausible error in the oracle must break some pin ----
# The test copies oracle.c, plants one mistake by text substitution, compiles the copy
# into a temporary library and checks that the pins above reject it.

# ---- SigLIP with a label matrix (several positives per row, extra negative columns)

def torch_siglip_labels(A, B, prefixes, t, b, weights, Z):
    """Per-prefix losses, dA, dB, d/dt and d/db of sum_k w_k L_k by torch autograd (float64),
    z = +1 where the label matrix Z is set, -1 elsewhere."""
    At = torch.tensor(A, dtype=torch.float64, requires_grad=True)
    Bt = torch.tensor(B, dtype=torch.float64, requires_grad=True)
    tt = torch.tensor(t, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    z = 2.0 * torch.tensor(Z, dtype=torch.float64) - 1.0
    losses, total = [], 0.0
    for p, w in zip(prefixes, weights):
        cos = F.normalize(At[:, :p], dim=1, eps=1e-30) @ F.normalize(Bt[:, :p], dim=1, eps=1e-30).T
        L = -F.logsigmoid(z * (tt * cos + bt)).sum() / At.shape[0]
        losses.append(L.item())
        total = total + w * L
    total.backward()
    return np.array(losses), At.grad.numpy(), Bt.grad.numpy(), tt.grad.item(), bt.grad.item()


def _labels(Na, Nb, seed):
    """Random CSR positives: up to three per row (one row has none), ids increasing."""
    rng = np.random.default_rng(seed)
    offsets, ids = [0], []
    for i in range(Na):
        k = 0 if i == 1 else int(rng.integers(1, 4))
        ids += sorted(rng.choice(Nb, size=k, replace=False).tolist())
        offsets.append(len(ids))
    return np.array(offsets), np.array(ids)


def test_labels_match_torch_autograd():
    rng = np.random.default_rng(23)
    Na, Nb, D, pre = 7, 11, 128, (32, 64, 128)
    a = rng.standard_normal((Na, D))
    b = rng.standard_normal((Nb, D))
    b[:Na] += a
    A, B = _bits(a), _bits(b)
    csr = _labels(Na, Nb, 5)
    Z = oracle.label_matrix(csr, Na, Nb)
    w = rng.uniform(0.5, 2.0, len(pre))
    t, bias = 4.0, -2.0
    got = oracle.fwd_bwd("siglip", A, B, pre, t, bias, w, labels=csr)
    ref = torch_siglip_labels(_wide(A), _wide(B), pre, t, bias, w, Z)
    np.testing.assert_allclose(got["loss"], ref[0], rtol=1e-12)
    np.testing.assert_allclose(got["dA"], ref[1], rtol=1e-9, atol=1e-13)
    np.testing.assert_allclose(got["dB"], ref[2], rtol=1e-9, atol=1e-13)
    ds, db = oracle.scale_grads("siglip", A, B, pre, t, bias, w, labels=csr)
    np.testing.assert_allclose([ds, db], ref[3:], rtol=1e-10, atol=1e-13)
    # the dense matrix and the CSR lists name the same pairs
    np.testing.assert_array_equal(oracle.fwd_bwd("siglip", A, B, pre, t, bias, w, labels=Z)["dA"], got["dA"])


def test_diagonal_labels_equal_the_default_positives():
    A, B = _random_pair(9, 128, 24)
    Z = np.eye(9, dtype=np.uint8)
    r0 = oracle.fwd_bwd("siglip", A, B, (64, 128), 10.0, -10.0)
    r1 = oracle.fwd_bwd("siglip", A, B, (64, 128), 10.0, -10.0, labels=Z)
    for k in r0:
        np.testing.assert_array_equal(r0[k], r1[k])


def test_labels_one_hot_closed_form():
    """One-hot rows: cos_ij = [i == j], so every cell's logit is t + b (diagonal) or b, and
    the loss counts positive / negative cells of each kind."""
    Na, Nb, D, t, b = 5, 9, 64, 6.0, -1.5
    E = np.eye(Nb, D)
    A, B = _bits(E[:Na]), _bits(E)
    csr = _labels(Na, Nb, 8)
    Z = oracle.label_matrix(csr, Na, Nb).astype(bool)
    sp = lambda y: np.log1p(np.exp(y))  # noqa: E731
    diag = np.zeros((Na, Nb), bool)
    diag[np.arange(Na), np.arange(Na)] = True
    n_pd, n_po = (Z & diag).sum(), (Z & ~diag).sum()
    n_nd, n_no = (~Z & diag).sum(), (~Z & ~diag).sum()
    L = (n_pd * sp(-(t + b)) + n_nd * sp(t + b) + n_po * sp(-b) + n_no * sp(b)) / Na
    got = oracle.fwd_bwd("siglip", A, B, (32, 64), t, b, labels=csr)
    np.testing.assert_allclose(got["loss"], [L, L], rtol=1e-13)
    # d/db: every cell's sigmoid minus one per positive
    sig = lambda y: 1.0 / (1.0 + np.exp(-y))  # noqa: E731
    dbias = 2 * (Na * sig(t + b) + (Na * Nb - Na) * sig(b) - Z.sum()) / Na
    assert abs(oracle.scale_grads("siglip", A, B, (32, 64), t, b, labels=csr)[1] - dbias) < 1e-13


# ---- the one-set loss (one set scored against itself, mirrored cells share labels)

def _sym_labels(N, seed):
    """Seeded symmetric positives between distinct rows: a few pairs and one triple."""
    rng = np.random.default_rng(seed)
    Z = np.zeros((N, N), np.uint8)
    perm = rng.permutation(N)
    for u in range(0, N - 1, 3):
        i, j = perm[u], perm[u + 1]
        Z[i, j] = Z[j, i] = 1
    i, j, k = perm[:3]
    Z[i, k] = Z[k, i] = 1
    return Z


def torch_oneset(X, prefixes, t, b, weights, Z):
    Xt = torch.tensor(X, dtype=torch.float64, requires_grad=True)
    tt = torch.tensor(t, dtype=torch.float64, requires_grad=True)
    bt = torch.tensor(b, dtype=torch.float64, requires_grad=True)
    N = Xt.shape[0]
    z = 2.0 * torch.tensor(Z, dtype=torch.float64) - 1.0
    off = 1.0 - torch.eye(N, dtype=torch.float64)
    losses, total = [], 0.0
    for p, w in zip(prefixes, weights):
        xn = F.normalize(Xt[:, :p], dim=1, eps=1e-30)
        L = -(F.logsigmoid(z * (tt * (xn @ xn.T) + bt)) * off).sum() / N
        losses.append(L.item())
        total = total + w * L
    total.backward()
    return np.array(losses), Xt.grad.numpy(), tt.grad.item(), bt.grad.item()


def test_oneset_matches_torch_autograd():
    rng = np.random.default_rng(31)
    N, D, pre = 9, 128, (32, 64, 128)
    X = _bits(rng.standard_normal((N, D)))
    Z = _sym_labels(N, 3)
    w = rng.uniform(0.5, 2.0, len(pre))
    t, b = 5.0, -2.5
    got = oracle.oneset(X, pre, t, b, Z, w)
    L, gX, gt, gb = torch_oneset(_wide(X), pre, t, b, w, Z)
    np.testing.assert_allclose(got["loss"], L, rtol=1e-12)
    np.testing.assert_allclose(got["dX"], gX, rtol=1e-9, atol=1e-13)
    np.testing.assert_allclose([got["dscale"], got["dbias"]], [gt, gb], rtol=1e-10, atol=1e-13)
    np.testing.assert_allclose(got["row_terms"].mean(axis=1), got["loss"], rtol=1e-13)


def test_oneset_is_the_two_set_loss_of_the_set_with_itself():
    """Both roles of every row: dX = dA + dB of the two-set loss at A = B = X, whose diagonal
    cells (cosine 1, no gradient) hold the only difference in the loss."""
    rng = np.random.default_rng(32)
    N, pre, t, b = 8, (64, 128), 4.0, -1.0
    X = _bits(rng.standard_normal((N, 128)))
    Z = _sym_labels(N, 4)
    one = oracle.oneset(X, pre, t, b, Z)
    two = oracle.fwd_bwd("siglip", X, X, pre, t, b, labels=Z)
    sp = lambda y: np.log1p(np.exp(y))  # noqa: E731
    diag = sp(t + b) * N / N  # every self-cell is a negative (Z has an empty diagonal) with x = t + b
    np.testing.assert_allclose(one["loss"], two["loss"] - diag, rtol=1e-12)
    np.testing.assert_allclose(one["dX"], two["dA"] + two["dB"], rtol=1e-9, atol=1e-13)


def test_oneset_identical_rows_closed_form():
    N, t, b = 6, 3.0, -1.0
    X = _bits(np.tile(np.random.default_rng(5).standard_normal(128), (N, 1)))
    Z = _sym_labels(N, 6)
    sp = lambda y: np.log1p(np.exp(y))  # noqa: E731
    pos = Z.sum(axis=1)
    L = np.sum(pos * sp(-(t + b)) + (N - 1 - pos) * sp(t + b)) / N
    got = oracle.oneset(X, (64, 128), t, b, Z)
    np.testing.assert_allclose(got["loss"], [L, L], rtol=1e-13)
    assert np.abs(got["dX"]).max() < 1e-12


def test_oneset_finite_differences():
    rng = np.random.default_rng(33)
    N, D, pre = 5, 16, (8, 16)
    X = rng.standard_normal((N, D))
    Z = _sym_labels(N, 7)
    w = np.array([0.6, 1.4])
    t, b = 2.0, -0.5
    got = oracle.oneset(X, pre, t, b, Z, w)

    def f(X_=X, t_=t, b_=b):
        return float(np.dot(w, oracle.oneset(X_, pre, t_, b_, Z, w, grads=False)["loss"]))

    h = 1e-6
    for (i, d) in ((0, 3), (2, 9), (4, 15)):
        Xp, Xm = X.copy(), X.copy()
        Xp[i, d] += h
        Xm[i, d] -= h
        np.testing.assert_allclose(got["dX"][i, d], (f(Xp) - f(Xm)) / (2 * h), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(got["dscale"], (f(t_=t + h) - f(t_=t - h)) / (2 * h), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(got["dbias"], (f(b_=b + h) - f(b_=b - h)) / (2 * h), rtol=1e-6, atol=1e-9)


MUTATIONS = {
    "dropped_projection_term": (
        "out[d] += g * (B[j * D + d] * rb[j] - c * A[i * D + d] * ra[i]) * ra[i];",
        "out[d] += g * (B[j * D + d] * rb[j]) * ra[i];"),
    "siglip_label_sign": ("double z = pos ? 1.0 : -1.0;", "double z = pos ? -1.0 : 1.0;"),
    "oneset_second_argument_dropped": (
        "out[d] += (g1 + g2) * (X[j * D + d] * r[j] - c * X[i * D + d] * r[i]) * r[i];",
        "out[d] += (g1) * (X[j * D + d] * r[j] - c * X[i * D + d] * r[i]) * r[i];"),
    "oneset_self_cell_counted": ("if (j == i) { /* a row is not paired with itself */",
                                 "if (j == i && 0) { /* a row is not paired with itself */"),
    "labels_ignored": ("return Z ? Z[i * Nb + j] != 0 : i == j;", "return i == j;"),
    "labels_row_shifted": ("return Z ? Z[i * Nb + j] != 0 : i == j;",
                           "return Z ? Z[((i + 1) % (Nb < 2 ? 1 : 2)) * Nb + j] != 0 : i == j;"),
    "column_lse_transposed": (
        "for (int64_t i = 0; i < Na; ++i) s += exp(tau * C[i * Nb + j] - m);",
        "for (int64_t i = 0; i < Na; ++i) s += exp(tau * C[j * Nb + i] - m);"),
    "prefix_off_by_one": ("for (int d = 0; d < p; ++d) dot += A[i * D + d] * B[j * D + d];",
                          "for (int d = 0; d < p - 1; ++d) dot += A[i * D + d] * B[j * D + d];"),
    "clip_normaliser": ("L = 0.5 * (Lr / N + Lc / N);", "L = (Lr / N + Lc / N);"),
    "dB_wrong_norm": ("out[d] += g * (A[i * D + d] * ra[i] - c * B[j * D + d] * rb[j]) * rb[j];",
                      "out[d] += g * (A[i * D + d] * ra[i] - c * B[j * D + d] * rb[j]) * ra[i];"),
    "dscale_column_half_dropped": ("gk = 0.5 * (rows / (double)Na + cols / (double)Nb);",
                                   "gk = 0.5 * (rows / (double)Na);"),
    "dscale_positive_sign": (
        "const double g = sigmoid(t * C[i * Nb + j] + bias) - (positive(Z, Nb, i, j) ? 1.0 : 0.0);",
        "const double g = sigmoid(t * C[i * Nb + j] + bias) + (positive(Z, Nb, i, j) ? 1.0 : 0.0);"),
}


def _pins_pass():
    """Run the cheap pins; return False as soon as one fails."""
    checks = [
        lambda: test_matches_torch_library_and_autograd(*CASES[0]),
        lambda: test_matches_torch_library_and_autograd(*CASES[1]),
        test_identical_embeddings_closed_forms,
        test_one_hot_orthogonal_closed_forms,
        lambda: test_scale_grads_match_autograd(*CASES[0]),
        lambda: test_scale_grads_match_autograd(*CASES[1]),
        test_labels_match_torch_autograd,
        test_oneset_matches_torch_autograd,
    ]
    for c in checks:
        try:
            c()
        except AssertionError:
            return False
    return True


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes_are_caught(name, tmp_path):
    import subprocess

    old, new = MUTATIONS[name]
    src = open(oracle.ref._SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", str(path), "-o", str(so), "-lm"])
    with oracle.ref.use_library(str(so)):
        assert not _pins_pass(), f"planted mistake {name} was not caught"
    assert _pins_pass()
