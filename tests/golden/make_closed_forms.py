"""Write closed_forms_prefix_ladder.txt: exact losses of the "prefix ladder" embeddings.

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


if __name__ == "__main__":
    main()
