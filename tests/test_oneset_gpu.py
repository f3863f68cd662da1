"""The one-set SigLIP loss (one set scored against itself, mirrored cells share labels)
on the GPU against the float64 oracle: loss relative error <= 2e-3, gradient max-abs
<= 1e-2 * max|grad|, like the other parity tests."""
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


def pair_set(N, D, noise, seed, extra=0):
    """An interleaved set of pairs (rows 2m and 2m + 1 are an embedding and its noisy
    partner, as an image and its caption), labelled as positive pairs, plus `extra` seeded
    symmetric positives between other rows; an odd N leaves the last row unpaired."""
    a, b = synth.paired((N + 1) // 2, D, noise, seed)
    X = np.empty((N, D), np.uint16)
    X[0::2] = a[: (N + 1) // 2]
    X[1::2] = b[: N // 2]
    Z = np.zeros((N, N), bool)
    for m in range(N // 2):
        Z[2 * m, 2 * m + 1] = Z[2 * m + 1, 2 * m] = True
    rng = np.random.default_rng(seed)
    for _ in range(extra):
        i, j = rng.choice(N, 2, replace=False)
        Z[i, j] = Z[j, i] = True
    offsets = np.concatenate([[0], np.cumsum(Z.sum(axis=1))]).astype(np.int64)
    ids = np.nonzero(Z)[1].astype(np.int32)  # row-major: each row's ids increasing
    return X, (offsets, ids)


def run(binding, X16, labels, pre, t, b, weights=None, workspace=None, grads=True, expect_status=0):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.oneset_fwd_bwd(dev(X16), labels, pre, t, b, weights, grads=grads, terms=True, workspace=workspace,
                                 device_status=status, scale_grads=grads)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def check(got, ref, grads=True):
    rel = np.abs(got["loss"] - ref["loss"]) / np.abs(ref["loss"])
    assert rel.max() <= LOSS_RTOL, f"loss {got['loss']} vs oracle {ref['loss']}"
    terr = np.abs(got["row_terms"] - ref["row_terms"]).max()
    assert terr <= LOSS_RTOL * np.abs(ref["row_terms"]).max(), f"row terms err {terr:.3e}"
    if grads:
        err = np.abs(got["dX"] - ref["dX"]).max()
        assert err <= GRAD_FRAC * np.abs(ref["dX"]).max(), f"dX: err {err:.3e} vs max {np.abs(ref['dX']).max():.3e}"
        assert abs(got["d_logit_scale"][0] - ref["dscale"]) <= 1e-2 * abs(ref["dscale"]) + 1e-6
        assert abs(got["d_bias"][0] - ref["dbias"]) <= 1e-2 * abs(ref["dbias"]) + 1e-6


CASES = [
    # N, D, prefixes, t, b, noise, seed, extra positives
    (300, 1024, LADDER, 10.0, -10.0, 0.7, 121, 20),
    (513, 1024, LADDER, 4.0, -2.0, 0.7, 122, 0),          # ragged, one unpaired row
    (257, 640, (128, 320, 512), 6.0, -3.0, 0.8, 123, 40),
    (2, 1024, LADDER, 10.0, -10.0, 0.7, 124, 0),          # one pair
]


@pytest.mark.parametrize("N,D,pre,t,b,noise,seed,extra", CASES)
def test_parity_oneset(ctx, N, D, pre, t, b, noise, seed, extra):
    X16, labels = pair_set(N, D, noise, seed, extra)
    w = list(np.linspace(0.5, 1.5, len(pre)))
    got = run(ctx, X16, labels, pre, t, b, weights=w)
    ref = oracle.oneset(X16, pre, t, b, labels, w)
    check(got, ref)
    check(run(ctx, X16, labels, pre, t, b, weights=w, grads=False), ref, grads=False)


def test_oneset_smallest_workspace(ctx):
    N, D = 640, 1024
    X16, labels = pair_set(N, D, 0.7, 125, 10)
    k = ctx.KINDS["siglip"]
    wmin = ctx.uf_contrastive_workspace_min(N, N, D, LADDER, k, True)
    assert wmin < ctx.uf_contrastive_workspace_size(N, N, D, LADDER, k, True)
    got = run(ctx, X16, labels, LADDER, 10.0, -10.0, workspace=torch.empty(wmin, dtype=torch.uint8, device="cuda"))
    check(got, oracle.oneset(X16, LADDER, 10.0, -10.0, labels))


def test_oneset_device_scalars(ctx):
    X16, labels = pair_set(300, 1024, 0.7, 126, 5)
    t = torch.tensor([10.0], device="cuda")
    b = torch.tensor([-10.0], device="cuda")
    got = run(ctx, X16, labels, LADDER, t, b)
    check(got, oracle.oneset(X16, LADDER, 10.0, -10.0, labels))


@pytest.mark.parametrize("what", ["asymmetric", "self_pair"])
def test_oneset_malformed_labels_are_reported(ctx, what):
    N = 64
    X16, (offsets, ids) = pair_set(N, 1024, 0.7, 127, 0)
    Z = np.zeros((N, N), bool)
    for i in range(N):
        Z[i, ids[offsets[i]:offsets[i + 1]]] = True
    if what == "asymmetric":
        Z[0, 5] = True      # (0, 5) without (5, 0)
    else:
        Z[3, 3] = True
    offsets = np.concatenate([[0], np.cumsum(Z.sum(axis=1))]).astype(np.int64)
    ids = np.nonzero(Z)[1].astype(np.int32)
    run(ctx, X16, (offsets, ids), LADDER, 10.0, -10.0, expect_status=1)
