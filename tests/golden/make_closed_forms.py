"""Write closed_forms_prefix_ladder.txt and closed_forms_prefix_ladder_grads.txt: exact losses
and gradient entries of the "prefix ladder" embeddings.

The values come from the loss definitions alone, evaluated with mpmath at 40 digits.  Neither
the oracle nor the library is used.  Source of the definitions: "Scaling-Up Contrastive
Learning over NVLink Multicast", section "One Set or Two":
- CLIP turns each row of cosines into a softmax over the batch (symmetric: rows and columns);
- SigLIP is -(1/N) sum_ij log sigmoid(z_ij (t cos_ij + b)), with z = +1 on positives and -1
  elsewhere;
- the Matryoshka prefixes are the first 64, 128, 256, 512 and 1024 dimensions, each
  normalised on its own.

The embeddings, identical for A and B: row i (i < N <= 64) is one-hot at dimension i within
[0, 64), then 0.125 in every dimension of [64, 1024).  Every entry is exact in bf16.  At prefix p:
- the squared norm is 1 + s_p, with s_p = (p - 64) / 64;
- the diagonal cosine is 1;
- every off-diagonal cosine is kappa_p = s_p / (1 + s_p), i.e. 0, 1/2, 3/4, 7/8, 15/16.

Closed forms, per prefix:
- CLIP (and ROWS, the row half, queries = the first Nq rows): log(1 + (N - 1) e^{-tau (1 - kappa)});
- SigLIP: softplus(-(t + b)) + (N - 1) softplus(t kappa + b).

Run: python tests/golden/make_closed_forms.py
"""
import os

import mpmath as mp

mp.mp.dps = 40
PREFIXES = (64, 128, 256, 512, 1024)
OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms_prefix_ladder.txt")
OUT_GRAD = os.path.join(os.path.dirname(os.path.abspath(__file__)), "closed_forms_prefix_ladder_grads.txt")


def kappa(p):
    s = mp.mpf(p - 64) / 64
    return s / (1 + s)


def softplus(x):
    return mp.log1p(mp.exp(x))


def clip_like(n_cols, tau, p):
    return mp.log1p((n_cols - 1) * mp.exp(-mp.mpf(tau) * (1 - kappa(p))))


def siglip(n_cols, t, b, p):
    t, b = mp.mpf(t), mp.mpf(b)
    return softplus(-(t + b)) + (n_cols - 1) * softplus(t * kappa(p) + b)


CASES = [  # kind, rows (A), cols (B), scale, bias
    ("clip", 48, 48, 1 / 0.07, 0.0),
    ("clip", 48, 48, 100.0, 0.0),
    ("rows", 16, 48, 20.0, 0.0),
    ("siglip", 48, 48, 10.0, -10.0),
    ("siglip", 33, 33, 4.0, -2.0),
]


def grad_entry(kind, na, nb, sc, bias, i, d):
    """dA[i, d] of sum_k L_k (unit weights) for the ladder, by the chain rule through the
    normalisation, dL/da_i = (1/|a_i|) (sum_j g_ij b^_j - (sum_j g_ij cos_ij) a^_i) with
    g_ij = dL/dcos_ij.

    At prefix p, with s = s_p, k = kappa_p and q = 1 / (1 + s), the (shared) g are:
    - CLIP (A = B: rows and columns alike): g_ii = (tau/N)(pi - 1), g_ij = (tau/N)(1 - pi)/(N - 1),
      where pi = e^tau / (e^tau + (N-1) e^{tau k});
    - ROWS (Nq queries, Nk keys): the same with tau/Nq and N = Nk;
    - SigLIP: g_ii = -(t/N) alpha, g_ij = (t/N) beta, where alpha = sigmoid(-(t + b)) and
      beta = sigmoid(t k + b).
    The components of dA[i] are then, for the one-hot dimension of row i, for the one-hot
    dimension of another row j' < cols, and for a dimension in [64, p):
        q (g_ii - G),  q g_ij,  c q ((g_ii + (cols - 1) g_ij) - G),
    where G = g_ii + (cols - 1) g_ij k (the sum of g cos) and c = 0.125.  A dimension in
    [cols, 64) or beyond p receives nothing from prefix p."""
    tot = mp.mpf(0)
    c = mp.mpf("0.125")
    for p in PREFIXES:
        if d >= p:
            continue
        s = mp.mpf(p - 64) / 64
        k = s / (1 + s)
        q = 1 / (1 + s)
        if kind == "siglip":
            t, b = mp.mpf(sc), mp.mpf(bias)
            alpha = 1 / (1 + mp.exp(t + b))
            beta = 1 / (1 + mp.exp(-(t * k + b)))
            gii, gij, ncols = -(t / na) * alpha, (t / na) * beta, nb
        else:
            tau = mp.mpf(sc)
            ncols = nb
            pi = mp.exp(tau) / (mp.exp(tau) + (ncols - 1) * mp.exp(tau * k))
            gii, gij = (tau / na) * (pi - 1), (tau / na) * (1 - pi) / (ncols - 1)
        G = gii + (ncols - 1) * gij * k
        if d == i:  # row i's one-hot dimension: b^_i[d] = a^_i[d] = sqrt(q)
            tot += q * (gii - G)
        elif d < 64 and d < ncols:  # another row's one-hot dimension
            tot += q * gij
        elif 64 <= d:
            tot += c * q * ((gii + (ncols - 1) * gij) - G)
    return tot


GRAD_POINTS = [(0, 0), (0, 1), (0, 40), (0, 63), (0, 100), (0, 300), (0, 700), (5, 5), (5, 0)]


def main():
    lines = [
        "# Closed-form losses of the prefix-ladder embeddings (see make_closed_forms.py for the",
        "# construction and the derivation).  Source of the loss definitions: \"Scaling-Up",
        "# Contrastive Learning over NVLink Multicast\", section \"One Set or Two\".",
        "# columns: kind rows cols scale bias prefix loss",
    ]
    for kind, na, nb, sc, bias in CASES:
        for p in PREFIXES:
            v = siglip(nb, sc, bias, p) if kind == "siglip" else clip_like(nb, sc, p)
            lines.append(f"{kind} {na} {nb} {sc!r} {bias!r} {p} {mp.nstr(v, 20)}")
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    glines = [
        "# Closed-form gradient entries dA[i, d] of sum_k L_k (unit prefix weights) for the prefix-ladder",
        "# embeddings; derivation in make_closed_forms.py (grad_entry).  Source of the loss definitions:",
        "# \"Scaling-Up Contrastive Learning over NVLink Multicast\", section \"One Set or Two\".",
        "# columns: kind rows cols scale bias i d dA",
    ]
    for kind, na, nb, sc, bias in CASES:
        for i, d in GRAD_POINTS:
            if i >= na:
                continue
            v = grad_entry(kind, na, nb, sc, bias, i, d)
            glines.append(f"{kind} {na} {nb} {sc!r} {bias!r} {i} {d} {mp.nstr(v, 20)}")
    with open(OUT_GRAD, "w") as f:
        f.write("\n".join(glines) + "\n")


if __name__ == "__main__":
    main()
