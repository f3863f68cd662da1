"""Seeded synthetic embedding batches, as bf16 bit patterns.

This module only *draws* inputs; it contains none of the loss arithmetic, so that
the float64 oracle and the CUDA path can both consume exactly the same bf16 bits.

Recipe (all draws are float64 from numpy's PCG64; every matrix is rounded to bf16
once, at the end, with round-to-nearest-even done here in exact float64 arithmetic):

* ``paired(N, D, noise, seed)``: A_i ~ N(0, 1)^D, B_i = A_i + noise * eps_i.
  The two streams (A and eps) come from two children of ``SeedSequence(seed)``,
  so chunked generation gives the same numbers as one big draw.
* ``paired_hard(N, D, noise, dup_frac, dup_noise, seed)``: as ``paired``, then
  ``floor(dup_frac * N)`` rows H (chosen without replacement) are replaced by
  near-duplicates of a source row k not in H: A_i = A_k + dup_noise * eps',
  B_i = B_k + dup_noise * eps'' (fresh draws), so B_k becomes a hard negative of A_i.
* ``queries_keys(Nq, Nk, D, noise, seed)``: keys_j ~ N(0, 1)^D,
  query_i = key_i + noise * eps_i for i < Nq (the first Nq keys are the positives).

The workloads follow the five benchmark configurations of the Matryoshka contrastive
loss (prefixes 64..1024 of D = 1024): CLIP N=256 and N=4096 with noise 1.0, SigLIP
N=16384 with noise 0.7, CLIP N=65536 with 10% near-duplicate hard negatives, and
row-direction InfoNCE with 8192 queries against 262144 keys with noise 0.8.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "round_to_bf16_bits",
    "bf16_bits_to_float",
    "paired",
    "paired_hard",
    "queries_keys",
    "prefix_ladder",
    "workload",
    "WORKLOADS",
]

_CHUNK_ROWS = 8192


def round_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even); return uint16 bits.

    Done in exact float64 arithmetic: |x| = m * 2**e with m in [0.5, 1); bf16 keeps
    8 significant bits, so the rounded value is rint(m * 256) * 2**(e - 8), which
    float64 holds exactly. ``np.rint`` rounds halves to even. The exact bf16 value
    is then also an exact float32, whose top 16 bits are the bf16 pattern.
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)
    r = np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)
    if np.any(np.abs(r[r != 0]) < np.finfo(np.float32).tiny) or np.any(~np.isfinite(r)):
        raise ValueError("value outside the normal bf16 range")
    return (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) exactly to float32."""
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _streams(seed: int, n: int):
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def paired(N: int, D: int, noise: float, seed: int):
    """A, B as uint16 bf16 bits of shape (N, D): B = A + noise * eps."""
    ga, ge = _streams(seed, 2)
    A = np.empty((N, D), np.uint16)
    B = np.empty((N, D), np.uint16)
    for r0 in range(0, N, _CHUNK_ROWS):
        r1 = min(N, r0 + _CHUNK_ROWS)
        a = ga.standard_normal((r1 - r0, D))
        b = a + noise * ge.standard_normal((r1 - r0, D))
        A[r0:r1] = round_to_bf16_bits(a)
        B[r0:r1] = round_to_bf16_bits(b)
    return A, B


def prefix_ladder(N: int, D: int = 1024):
    """The prefix-ladder batch as bf16 bits (N <= 64 rows, D > 64): row i is one-hot at
    dimension i within [0, 64), then 0.125 in every dimension of [64, D).  Every entry is
    exact in bf16, and every off-diagonal cosine at a prefix p is the same number, so the
    losses have closed forms (tests/golden/make_closed_forms.py)."""
    if not 1 <= N <= 64 or D <= 64:
        raise ValueError("the prefix ladder needs 1 <= N <= 64 and D > 64")
    x = np.zeros((N, D))
    x[np.arange(N), np.arange(N)] = 1.0
    x[:, 64:] = 0.125
    return round_to_bf16_bits(x)


def paired_hard(N: int, D: int, noise: float, dup_frac: float, dup_noise: float, seed: int):
    """``paired`` plus near-duplicate rows that act as hard negatives (see module doc)."""
    ga, ge, gh = _streams(seed, 3)
    a_all = np.empty((N, D), np.float64)
    b_all = np.empty((N, D), np.float64)
    for r0 in range(0, N, _CHUNK_ROWS):
        r1 = min(N, r0 + _CHUNK_ROWS)
        a = ga.standard_normal((r1 - r0, D))
        a_all[r0:r1] = a
        b_all[r0:r1] = a + noise * ge.standard_normal((r1 - r0, D))
    n_dup = int(np.floor(dup_frac * N))
    H = gh.choice(N, size=n_dup, replace=False)
    is_dup = np.zeros(N, bool)
    is_dup[H] = True
    pool = np.flatnonzero(~is_dup)
    src = pool[gh.integers(0, pool.size, size=n_dup)]
    for i, k in zip(H, src):
        a_all[i] = a_all[k] + dup_noise * gh.standard_normal(D)
        b_all[i] = b_all[k] + dup_noise * gh.standard_normal(D)
    A = np.empty((N, D), np.uint16)
    B = np.empty((N, D), np.uint16)
    for r0 in range(0, N, _CHUNK_ROWS):
        r1 = min(N, r0 + _CHUNK_ROWS)
        A[r0:r1] = round_to_bf16_bits(a_all[r0:r1])
        B[r0:r1] = round_to_bf16_bits(b_all[r0:r1])
    return A, B


def queries_keys(Nq: int, Nk: int, D: int, noise: float, seed: int):
    """Q (Nq, D) and K (Nk, D) bf16 bits: query_i = key_i + noise * eps_i."""
    gk, ge = _streams(seed, 2)
    Kb = np.empty((Nk, D), np.uint16)
    Qb = np.empty((Nq, D), np.uint16)
    for r0 in range(0, Nk, _CHUNK_ROWS):
        r1 = min(Nk, r0 + _CHUNK_ROWS)
        k = gk.standard_normal((r1 - r0, D))
        Kb[r0:r1] = round_to_bf16_bits(k)
        if r0 < Nq:
            q1 = min(r1, Nq)
            q = k[: q1 - r0] + noise * ge.standard_normal((q1 - r0, D))
            Qb[r0:q1] = round_to_bf16_bits(q)
    return Qb, Kb


# The five benchmark workloads: name -> (loss kind, generator, arguments, logit scale, bias)
WORKLOADS = {
    "clip_n256": dict(kind="clip", gen="paired", N=256, D=1024, noise=1.0, seed=0, scale=1 / 0.07, bias=0.0),
    "clip_n4096": dict(kind="clip", gen="paired", N=4096, D=1024, noise=1.0, seed=1, scale=1 / 0.07, bias=0.0),
    "siglip_n16384": dict(kind="siglip", gen="paired", N=16384, D=1024, noise=0.7, seed=2, scale=10.0, bias=-10.0),
    "clip_n65536_hardneg": dict(kind="clip", gen="paired_hard", N=65536, D=1024, noise=1.0, seed=3,
                                scale=1 / 0.07, bias=0.0, dup_frac=0.1, dup_noise=0.05),
    "rows_q8192_k262144": dict(kind="rows", gen="queries_keys", Nq=8192, Nk=262144, D=1024, noise=0.8, seed=4,
                               scale=1 / 0.05, bias=0.0),
}
PREFIXES = (64, 128, 256, 512, 1024)


def workload(name: str):
    """Return (kind, A_bits, B_bits, scale, bias) for one of ``WORKLOADS``."""
    w = WORKLOADS[name]
    if w["gen"] == "paired":
        A, B = paired(w["N"], w["D"], w["noise"], w["seed"])
    elif w["gen"] == "paired_hard":
        A, B = paired_hard(w["N"], w["D"], w["noise"], w["dup_frac"], w["dup_noise"], w["seed"])
    else:
        A, B = queries_keys(w["Nq"], w["Nk"], w["D"], w["noise"], w["seed"])
    return w["kind"], A, B, w["scale"], w["bias"]
