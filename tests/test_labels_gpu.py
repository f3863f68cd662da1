"""SigLIP with explicit positives (CSR lists, several per row or none) and with extra
negative columns (Nb > Na): parity of the CUDA path with the float64 oracle, under the
tolerances of the other parity tests (loss relative error <= 2e-3, gradients max-abs
<= 1e-2 * max|grad|)."""
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


def csr_labels(Na, Nb, seed, max_pos=3, diag=True):
    """Seeded positives: up to max_pos per row (some rows none), the row's own column
    among them when diag, ids increasing."""
    rng = np.random.default_rng(seed)
    offsets, ids = [0], []
    for i in range(Na):
        k = int(rng.integers(0, max_pos + 1))
        cols = set(rng.choice(Nb, size=k, replace=False).tolist())
        if diag and k:
            cols.add(i)
        ids += sorted(cols)
        offsets.append(len(ids))
    return np.array(offsets, np.int64), np.array(ids, np.int32)


def run(binding, A16, B16, pre, t, b, labels=None, weights=None, workspace=None, scale_grads=True, grads=True,
        expect_status=0):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.contrastive_fwd_bwd(dev(A16), dev(B16), "siglip", pre, t, b, weights, grads=grads, terms=True,
                                      workspace=workspace, device_status=status,
                                      scale_grads=scale_grads and grads, labels=labels)
    torch.cuda.synchronize()
    assert int(status.item()) == expect_status
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def check(got, ref, grads=True):
    rel = np.abs(got["loss"] - ref["loss"]) / np.abs(ref["loss"])
    assert rel.max() <= LOSS_RTOL, f"loss {got['loss']} vs oracle {ref['loss']}"
    terr = np.abs(got["row_terms"] - ref["row_terms"]).max()
    assert terr <= LOSS_RTOL * np.abs(ref["row_terms"]).max(), f"row terms err {terr:.3e}"
    if grads:
        for g in ("dA", "dB"):
            err = np.abs(got[g] - ref[g]).max()
            assert err <= GRAD_FRAC * np.abs(ref[g]).max(), f"{g}: err {err:.3e} vs max {np.abs(ref[g]).max():.3e}"


def make(Na, Nb, D, seed, noise):
    a, b = synth.queries_keys(Na, Nb, D, noise, seed)  # key i is query i's partner, keys past Na extra
    return a, b


CASES = [
    # Na, Nb, D, prefixes, t, b, noise, seed, max positives per row
    (300, 300, 1024, LADDER, 10.0, -10.0, 0.7, 101, 3),
    (200, 700, 1024, LADDER, 4.0, -2.0, 0.7, 102, 4),     # extra negative columns
    (257, 400, 640, (128, 320, 512), 6.0, -3.0, 0.8, 103, 2),
    (1, 300, 1024, LADDER, 10.0, -10.0, 0.7, 104, 5),
]


@pytest.mark.parametrize("Na,Nb,D,pre,t,b,noise,seed,maxp", CASES)
def test_parity_labelled_positives(ctx, Na, Nb, D, pre, t, b, noise, seed, maxp):
    A16, B16 = make(Na, Nb, D, seed, noise)
    labels = csr_labels(Na, Nb, seed, maxp)
    w = list(np.linspace(1.5, 0.5, len(pre)))
    got = run(ctx, A16, B16, pre, t, b, labels=labels, weights=w)
    ref = oracle.fwd_bwd("siglip", A16, B16, pre, t, b, w, labels=labels)
    check(got, ref)
    ds, db = oracle.scale_grads("siglip", A16, B16, pre, t, b, w, labels=labels)
    assert abs(got["d_logit_scale"][0] - ds) <= 1e-2 * abs(ds) + 1e-6
    assert abs(got["d_bias"][0] - db) <= 1e-2 * abs(db) + 1e-6
    fwd = run(ctx, A16, B16, pre, t, b, labels=labels, weights=w, grads=False)  # the forward-only pass
    check(fwd, ref, grads=False)


def test_labels_with_the_smallest_workspace(ctx):
    Na, Nb, D = 300, 500, 1024
    A16, B16 = make(Na, Nb, D, 105, 0.7)
    labels = csr_labels(Na, Nb, 105, 3)
    k = ctx.KINDS["siglip"]
    wmin = ctx.uf_contrastive_workspace_min(Na, Nb, D, LADDER, k, True)
    assert wmin < ctx.uf_contrastive_workspace_size(Na, Nb, D, LADDER, k, True)
    ws = torch.empty(wmin, dtype=torch.uint8, device="cuda")
    got = run(ctx, A16, B16, LADDER, 10.0, -10.0, labels=labels, workspace=ws)
    check(got, oracle.fwd_bwd("siglip", A16, B16, LADDER, 10.0, -10.0, labels=labels))


def test_diagonal_labels_match_the_default_positives(ctx):
    A16, B16 = make(300, 300, 1024, 106, 0.7)
    eye = (np.arange(301, dtype=np.int64), np.arange(300, dtype=np.int32))
    ref = oracle.fwd_bwd("siglip", A16, B16, LADDER, 10.0, -10.0)
    check(run(ctx, A16, B16, LADDER, 10.0, -10.0, labels=eye), ref)
    check(run(ctx, A16, B16, LADDER, 10.0, -10.0), ref)


def test_extra_negative_columns_without_labels(ctx):
    A16, B16 = make(200, 700, 1024, 107, 0.7)
    got = run(ctx, A16, B16, LADDER, 10.0, -10.0)
    check(got, oracle.fwd_bwd("siglip", A16, B16, LADDER, 10.0, -10.0))


def test_no_positives_at_all(ctx):
    A16, B16 = make(128, 256, 1024, 108, 0.7)
    labels = (np.zeros(129, np.int64), np.zeros(0, np.int32))
    got = run(ctx, A16, B16, LADDER, 4.0, -1.0, labels=labels)
    check(got, oracle.fwd_bwd("siglip", A16, B16, LADDER, 4.0, -1.0, labels=labels))


@pytest.mark.parametrize("what", ["id_out_of_range", "ids_not_increasing", "offsets_decreasing"])
def test_malformed_labels_are_reported(ctx, what):
    # every bad entry stays inside the arrays handed over; the kernels skip it and report
    Na, Nb = 64, 128
    A16, B16 = make(Na, Nb, 1024, 109, 0.7)
    offsets, ids = csr_labels(Na, Nb, 109, 3)
    offsets, ids = offsets.copy(), ids.copy()
    if what == "id_out_of_range":
        ids[0] = Nb
    elif what == "ids_not_increasing":
        r = int(np.argmax(np.diff(offsets) >= 2))
        ids[offsets[r]:offsets[r] + 2] = ids[offsets[r]]
    else:
        assert offsets[5] >= 1
        offsets[6] = offsets[5] - 1  # row 5 ends before it starts
    run(ctx, A16, B16, LADDER, 10.0, -10.0, labels=(offsets, ids), expect_status=1)
