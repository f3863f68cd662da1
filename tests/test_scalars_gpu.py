"""The loss's learned scalars on the GPU: large logit scales (the max-shifted statistics),
scales and biases read from device memory, and a captured CUDA graph that follows a scale
updated in place.  Parity with the float64 oracle under the same tolerances as the other
parity tests (loss relative error <= 2e-3, gradients max-abs <= 1e-2 * max|grad|)."""
import numpy as np
import pytest

import oracle
from contrastive_embedding_loss_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LADDER = (64, 128, 256, 512, 1024)
LOSS_RTOL = 2e-3
GRAD_FRAC = 1e-2


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding

    assert binding.uf_contrastive_init(0) == 0
    return binding


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def scalar(v):
    return torch.tensor([v], dtype=torch.float32, device="cuda")


def make(kind, Na, Nb, D, seed, noise):
    if kind == "rows":
        return synth.queries_keys(Na, Nb, D, noise, seed)
    return synth.paired(Na, D, noise, seed)


def run(binding, kind, A16, B16, pre, scale, bias, weights=None, scale_grads=False, expect_status=0):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.contrastive_fwd_bwd(dev(A16), dev(B16), kind, pre, scale, bias, weights, grads=True, terms=True,
                                      device_status=status, scale_grads=scale_grads)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def check(got, ref, kind, tau):
    # the oracle's loss is LSE - s_ii, a difference of O(tau) float64 numbers: below about
    # 64 ulp(tau) it is rounding (it can even come out negative), so that is the floor
    floor = 64 * np.finfo(np.float64).eps * tau
    err = np.abs(got["loss"] - ref["loss"])
    assert np.all(err <= LOSS_RTOL * np.abs(ref["loss"]) + floor), f"loss {got['loss']} vs oracle {ref['loss']}"
    terr = np.abs(got["row_terms"] - ref["row_terms"]).max()
    assert terr <= LOSS_RTOL * np.abs(ref["row_terms"]).max(), f"row terms err {terr:.3e}"
    if kind == "clip":
        cerr = np.abs(got["col_terms"] - ref["col_terms"]).max()
        assert cerr <= LOSS_RTOL * np.abs(ref["col_terms"]).max(), f"col terms err {cerr:.3e}"
    for g in ("dA", "dB"):
        err = np.abs(got[g] - ref[g]).max()
        assert err <= GRAD_FRAC * np.abs(ref[g]).max(), f"{g}: err {err:.3e} vs max {np.abs(ref[g]).max():.3e}"


LARGE = [
    # kind, Na, Nb, D, prefixes, tau, noise, seed.  Noise 6 puts the positives' cosine near
    # 0.16: at tau = 100 every e^{s - tau} of a row is below e^-84, where the fixed shift
    # would lose the sums to fp32 underflow.  (With the positives' cosine near 0.7 the loss
    # at tau = 100 is about e^-60: nothing left to compare.)
    ("clip", 300, 300, 1024, LADDER, 100.0, 6.0, 81),
    ("clip", 640, 640, 1024, LADDER, 100.0, 5.0, 82),
    ("clip", 257, 257, 384, (64, 192, 384), 60.0, 3.0, 83),
    ("clip", 256, 256, 1024, LADDER, 256.0, 6.0, 84),       # the largest supported scale
    ("clip", 192, 192, 1024, LADDER, 40.5, 3.0, 85),        # just past the fixed-shift range
    ("rows", 200, 700, 1024, LADDER, 100.0, 6.0, 86),
    ("rows", 1, 300, 1024, LADDER, 150.0, 8.0, 87),
]


@pytest.mark.parametrize("kind,Na,Nb,D,pre,tau,noise,seed", LARGE)
def test_parity_large_logit_scale(ctx, kind, Na, Nb, D, pre, tau, noise, seed):
    A16, B16 = make(kind, Na, Nb, D, seed, noise)
    w = list(np.linspace(0.5, 1.5, len(pre)))
    got = run(ctx, kind, A16, B16, pre, tau, 0.0, weights=w)
    ref = oracle.fwd_bwd(kind, A16, B16, pre, tau, 0.0, w)
    check(got, ref, kind, tau)


def test_hard_negatives_at_the_clip_clamp(ctx):
    # near-duplicate rows (their partner is a hard negative) at tau = 100
    A16, B16 = synth.paired_hard(512, 1024, 4.0, 0.1, 0.05, 88)
    got = run(ctx, "clip", A16, B16, LADDER, 100.0, 0.0)
    check(got, oracle.fwd_bwd("clip", A16, B16, LADDER, 100.0, 0.0), "clip", 100.0)


@pytest.mark.parametrize("kind,tau,bias,noise", [("clip", 1 / 0.07, 0.0, 1.0), ("rows", 20.0, 0.0, 0.8),
                                                 ("clip", 100.0, 0.0, 6.0), ("siglip", 10.0, -10.0, 0.7)])
def test_device_scalars_match_the_oracle(ctx, kind, tau, bias, noise):
    Na, Nb = (200, 700) if kind == "rows" else (300, 300)
    A16, B16 = make(kind, Na, Nb, 1024, 90, noise)
    got = run(ctx, kind, A16, B16, LADDER, scalar(tau), scalar(bias), scale_grads=True)
    ref = oracle.fwd_bwd(kind, A16, B16, LADDER, tau, bias)
    check(got, ref, kind, tau)
    ds, db = oracle.scale_grads(kind, A16, B16, LADDER, tau, bias)
    assert abs(got["d_logit_scale"][0] - ds) <= 1e-2 * abs(ds) + 1e-6
    if kind == "siglip":
        assert abs(got["d_bias"][0] - db) <= 1e-2 * abs(db) + 1e-6
        # SigLIP needs no shift: a device-held t and b run the very same arithmetic
        host = run(ctx, kind, A16, B16, LADDER, tau, bias, scale_grads=True)
        for key in ("loss", "dA", "dB", "d_logit_scale", "d_bias"):
            assert np.array_equal(got[key], host[key]), key


def test_max_shifted_path_agrees_with_the_fixed_shift(ctx):
    # a device-held tau always takes the max-shifted path; at tau = 1/0.07 the fixed shift
    # is exact too, so the two paths differ by rounding only
    A16, B16 = make("clip", 640, 640, 1024, 91, 1.0)
    fixed = run(ctx, "clip", A16, B16, LADDER, 1 / 0.07, 0.0, scale_grads=True)
    shifted = run(ctx, "clip", A16, B16, LADDER, scalar(1 / 0.07), 0.0, scale_grads=True)
    np.testing.assert_allclose(shifted["loss"], fixed["loss"], rtol=1e-5)
    for g in ("dA", "dB"):
        assert np.abs(shifted[g] - fixed[g]).max() <= 2e-3 * np.abs(fixed[g]).max()
    np.testing.assert_allclose(shifted["d_logit_scale"], fixed["d_logit_scale"], rtol=1e-3)


def test_out_of_range_device_scale_is_reported(ctx):
    A16, B16 = make("clip", 256, 256, 1024, 92, 1.0)
    run(ctx, "clip", A16, B16, LADDER, scalar(-1.0), 0.0, expect_status=1)
    run(ctx, "clip", A16, B16, LADDER, scalar(300.0), 0.0, expect_status=1)
    run(ctx, "siglip", A16, B16, LADDER, scalar(70.0), scalar(-20.0), expect_status=1)


def test_captured_graph_follows_the_scale_in_device_memory(ctx):
    kind, Na, D = "clip", 384, 1024
    A16, B16 = make(kind, Na, Na, D, 93, 4.0)
    A, B = dev(A16), dev(B16)
    tau = scalar(1 / 0.07)
    k = ctx.KINDS[kind]
    ws = torch.empty(ctx.uf_contrastive_workspace_size(Na, Na, D, LADDER, k, True), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        ctx.contrastive_fwd_bwd(A, B, kind, LADDER, tau, 0.0, workspace=ws, scale_grads=True)  # warm-up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        out = ctx.contrastive_fwd_bwd(A, B, kind, LADDER, tau, 0.0, workspace=ws, scale_grads=True)
    for t in (1 / 0.07, 50.0, 100.0):
        tau.fill_(t)
        graph.replay()
        torch.cuda.synchronize()
        got = {key: v.double().cpu().numpy() for key, v in out.items()}
        ref = oracle.fwd_bwd(kind, A16, B16, LADDER, t, 0.0)
        check({**got, "row_terms": ref["row_terms"], "col_terms": ref["col_terms"]}, ref, kind, t)
        ds, _ = oracle.scale_grads(kind, A16, B16, LADDER, t, 0.0)
        assert abs(got["d_logit_scale"][0] - ds) <= 1e-2 * abs(ds) + 1e-6, t
