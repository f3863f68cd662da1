"""Stored fixtures under tests/golden.

- closed_forms_prefix_ladder.txt: exact losses of the prefix-ladder embeddings, derived from the
  loss definitions ("Scaling-Up Contrastive Learning over NVLink Multicast", section "One Set or
  Two") and evaluated with mpmath by tests/golden/make_closed_forms.py.  They pin the oracle,
  since no oracle code is involved.  On a GPU the library is checked against them directly.
  Each prefix sees a different off-diagonal cosine, so a prefix's normalisation that used
  another prefix's norm, or a dropped term, changes the values.
- oracle_small.json: the oracle's own outputs on three small seeded cases
  (tests/golden/make_oracle_fixtures.py), a regression guard for the oracle's arithmetic.
"""
import json
import os

import numpy as np
import pytest

import oracle
from contrastive_embedding_loss_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
LADDER = (64, 128, 256, 512, 1024)
EPS = np.finfo(np.float64).eps


def closed_form_cases():
    """[(kind, rows, cols, scale, bias, [loss per prefix])] from the closed-form fixture."""
    groups = {}
    with open(os.path.join(GOLDEN, "closed_forms_prefix_ladder.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            kind, na, nb, sc, bias, p, loss = line.split()
            key = (kind, int(na), int(nb), float(sc), float(bias))
            groups.setdefault(key, {})[int(p)] = float(loss)
    return [(*key, [v[p] for p in LADDER]) for key, v in groups.items()]


CASES = closed_form_cases()
IDS = [f"{c[0]}-{c[1]}x{c[2]}-s{c[3]:g}" for c in CASES]


def ladder_inputs(rows, cols):
    X = synth.prefix_ladder(max(rows, cols))
    return X[:rows], X[:cols]


def test_fixture_covers_every_kind():
    assert {c[0] for c in CASES} == {"clip", "rows", "siglip"}
    assert all(len(c[5]) == len(LADDER) for c in CASES)


@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_oracle_matches_the_closed_forms(case):
    kind, na, nb, sc, bias, want = case
    A, B = ladder_inputs(na, nb)
    got = oracle.fwd_bwd(kind, A, B, LADDER, sc, bias, grads=False)["loss"]
    # the oracle forms LSE - s_ii around s = scale: below a few ulp(scale) that is rounding
    floor = 64 * EPS * sc
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=floor)


def closed_form_grad_cases():
    """[(kind, rows, cols, scale, bias, [(i, d, dA[i, d])])] from the gradient fixture."""
    groups = {}
    with open(os.path.join(GOLDEN, "closed_forms_prefix_ladder_grads.txt")) as f:
        for line in f:
            if not line.strip() or line.startswith("#"):
                continue
            kind, na, nb, sc, bias, i, d, v = line.split()
            groups.setdefault((kind, int(na), int(nb), float(sc), float(bias)), []).append((int(i), int(d), float(v)))
    return [(*key, pts) for key, pts in groups.items()]


GRAD_CASES = closed_form_grad_cases()
GRAD_IDS = [f"{c[0]}-{c[1]}x{c[2]}-s{c[3]:g}" for c in GRAD_CASES]


@pytest.mark.parametrize("case", GRAD_CASES, ids=GRAD_IDS)
def test_oracle_matches_the_closed_form_gradients(case):
    kind, na, nb, sc, bias, pts = case
    A, B = ladder_inputs(na, nb)
    dA = oracle.fwd_bwd(kind, A, B, LADDER, sc, bias)["dA"]
    scale = np.abs(dA).max()
    for i, d, want in pts:
        np.testing.assert_allclose(dA[i, d], want, rtol=1e-10, atol=1e-12 * scale, err_msg=f"dA[{i},{d}]")


def test_oracle_reproduces_its_stored_outputs():
    with open(os.path.join(GOLDEN, "oracle_small.json")) as f:
        fx = json.load(f)
    for case in fx["cases"]:
        A, B = getattr(synth, case["generator"])(*case["args"])
        r = oracle.fwd_bwd(case["kind"], A, B, tuple(case["prefixes"]), case["scale"], case["bias"])
        np.testing.assert_allclose(r["loss"], case["loss"], rtol=1e-12, atol=0, err_msg=case["name"])
        for side in ("dA", "dB"):
            want = case[side]
            x = r[side]
            scale = np.abs(x).max()
            np.testing.assert_allclose(x.sum(), want["sum"], rtol=0, atol=1e-12 * scale * x.size,
                                       err_msg=f"{case['name']} {side}")
            np.testing.assert_allclose((x * x).sum(), want["sumsq"], rtol=1e-11, err_msg=f"{case['name']} {side}")
            for i, j, v in want["entries"]:
                np.testing.assert_allclose(x[i, j], v, rtol=1e-11, atol=1e-14 * scale,
                                           err_msg=f"{case['name']} {side}[{i},{j}]")


@pytest.mark.gpu
@pytest.mark.parametrize("case", CASES, ids=IDS)
def test_library_matches_the_closed_forms(case):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding

    kind, na, nb, sc, bias, want = case
    A, B = ladder_inputs(na, nb)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.contrastive_fwd_bwd(dev(A), dev(B), kind, LADDER, sc, bias, grads=True, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out["loss"].double().cpu().numpy()
    # loss tolerance 2e-3 relative; below 64 ulp(scale) (values down to 1e-42 here) the
    # reference itself is rounding, as in the oracle comparisons
    floor = 64 * EPS * sc
    assert np.all(np.abs(got - np.asarray(want)) <= 2e-3 * np.abs(want) + floor), f"{got} vs {want}"
    assert torch.isfinite(out["dA"]).all() and torch.isfinite(out["dB"]).all()


# Mistakes planted in the oracle's loss arithmetic that the closed forms alone must reject:
# (anchor, replacement) pairs applied to a copy of oracle.c built on the CPU.
LOSS_MUTATIONS = {
    "prefix_norm_uses_full_width": (
        "ra[i] = inv_norm(A + i * D, p);\n#pragma omp parallel for schedule(static)\n"
        "    for (int64_t j = 0; j < Nb; ++j) rb[j] = inv_norm(B + j * D, p);",
        "ra[i] = inv_norm(A + i * D, D);\n#pragma omp parallel for schedule(static)\n"
        "    for (int64_t j = 0; j < Nb; ++j) rb[j] = inv_norm(B + j * D, D);"),
    "prefix_off_by_one": ("for (int d = 0; d < p; ++d) dot += A[i * D + d] * B[j * D + d];",
                          "for (int d = 0; d < p - 1; ++d) dot += A[i * D + d] * B[j * D + d];"),
    "clip_normaliser": ("L = 0.5 * (Lr / N + Lc / N);", "L = (Lr / N + Lc / N);"),
    "siglip_label_sign": ("double z = pos ? 1.0 : -1.0;", "double z = pos ? -1.0 : 1.0;"),
}


@pytest.mark.parametrize("name", sorted(LOSS_MUTATIONS))
def test_closed_forms_catch_planted_mistakes(name, tmp_path):
    import subprocess

    old, new = LOSS_MUTATIONS[name]
    src = open(oracle.ref._SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", str(path), "-o", str(so), "-lm"])

    def all_pass():
        for case in CASES:
            try:
                test_oracle_matches_the_closed_forms(case)
            except AssertionError:
                return False
        return True

    with oracle.ref.use_library(str(so)):
        assert not all_pass(), f"planted mistake {name} was not caught by the closed forms"
    assert all_pass()


GRAD_MUTATIONS = {
    "dropped_projection_term": (
        "out[d] += g * (B[j * D + d] * rb[j] - c * A[i * D + d] * ra[i]) * ra[i];",
        "out[d] += g * (B[j * D + d] * rb[j]) * ra[i];"),
    "prefix_norm_uses_full_width": LOSS_MUTATIONS["prefix_norm_uses_full_width"],
}


@pytest.mark.parametrize("name", sorted(GRAD_MUTATIONS))
def test_closed_form_gradients_catch_planted_mistakes(name, tmp_path):
    import subprocess

    old, new = GRAD_MUTATIONS[name]
    src = open(oracle.ref._SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "oracle_mut.c"
    path.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    subprocess.check_call(["gcc", "-O2", "-fopenmp", "-shared", "-fPIC", str(path), "-o", str(so), "-lm"])

    def all_pass():
        for case in GRAD_CASES:
            try:
                test_oracle_matches_the_closed_form_gradients(case)
            except AssertionError:
                return False
        return True

    with oracle.ref.use_library(str(so)):
        assert not all_pass(), f"planted mistake {name} was not caught by the closed-form gradients"
    assert all_pass()
