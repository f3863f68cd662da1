"""Parity at the full benchmark sizes, in the launch configuration the benchmark times.

The oracle computes outputs one row at a time on seeded samples: per-row loss terms of 512
rows and columns, and 512 gradient rows of each side.  A gradient row of an InfoNCE loss
needs the softmax normalisers of every row (and for CLIP every column) of the batch; the
oracle's large-batch normaliser routine (float64 matmuls on the host cores) supplies them,
and the C oracle's row loops check it again on the sampled rows.  At N = 65536 the dA and
dB contractions run as two separate launches, as in the benchmark.  Properties that hold at
any size are checked as well: the per-row Euler identity sum_d x_d dL/dx_d = 0 of a
scale-invariant loss, the mean of the row terms equalling the loss, A <-> B swap symmetry.
"""
import numpy as np
import pytest

import oracle
from contrastive_embedding_loss_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LADDER = (64, 128, 256, 512, 1024)


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding

    assert binding.uf_contrastive_init(0) == 0
    return binding


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def run(binding, kind, A16, B16, scale, bias):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.contrastive_fwd_bwd(dev(A16), dev(B16), kind, LADDER, scale, bias, grads=True, terms=True,
                                      device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out


def sample(n, k, seed):
    return np.sort(np.random.default_rng(seed).choice(n, size=min(k, n), replace=False))


def check_terms(got, ref, what):
    err = np.abs(got - ref).max()
    assert err <= 2e-3 * np.abs(ref).max(), f"{what}: err {err:.3e} vs max {np.abs(ref).max():.3e}"


def check_grad_rows(got, ref, what):
    err = np.abs(got - ref).max()
    assert err <= 1e-2 * np.abs(ref).max(), f"{what}: err {err:.3e} vs max {np.abs(ref).max():.3e}"


def check_loss_is_mean_of_terms(out, kind):
    loss = out["loss"].double().cpu().numpy()
    rt = out["row_terms"].double().mean(dim=1).cpu().numpy()
    if kind == "clip":
        rt = 0.5 * (rt + out["col_terms"].double().mean(dim=1).cpu().numpy())
    np.testing.assert_allclose(loss, rt, rtol=1e-5)


def check_euler(X16, G, what):
    x = torch.from_numpy(synth.bf16_bits_to_float(X16)).cuda().double()
    g = G.double()
    dot = (x * g).sum(dim=1).abs()
    bound = 2e-3 * x.norm(dim=1) * g.norm(dim=1) + 1e-30
    frac = (dot / bound).max().item()
    assert frac <= 1.0, f"{what}: Euler identity off by {frac:.2f} x tolerance"


def test_clip_n4096_full_oracle(ctx):
    kind, A16, B16, s, b = synth.workload("clip_n4096")
    out = run(ctx, kind, A16, B16, s, b)
    ref = oracle.fwd_bwd(kind, A16, B16, LADDER, s, b)
    got = {k: v.double().cpu().numpy() for k, v in out.items()}
    assert (np.abs(got["loss"] - ref["loss"]) / ref["loss"]).max() <= 2e-3
    check_terms(got["row_terms"], ref["row_terms"], "row terms")
    check_terms(got["col_terms"], ref["col_terms"], "col terms")
    check_grad_rows(got["dA"], ref["dA"], "dA")
    check_grad_rows(got["dB"], ref["dB"], "dB")


def test_siglip_n16384_sampled(ctx):
    kind, A16, B16, s, b = synth.workload("siglip_n16384")
    out = run(ctx, kind, A16, B16, s, b)
    check_loss_is_mean_of_terms(out, kind)
    rows = sample(A16.shape[0], 512, 1)
    ref_terms = oracle.row_terms_sampled(kind, A16, B16, LADDER, s, b, rows)
    check_terms(out["row_terms"][:, rows].double().cpu().numpy(), ref_terms, "row terms")
    gA = oracle.grad_rows(kind, True, A16, B16, LADDER, s, b, rows)
    check_grad_rows(out["dA"][rows].double().cpu().numpy(), gA, "dA rows")
    cols = sample(B16.shape[0], 512, 2)
    gB = oracle.grad_rows(kind, False, B16, A16, LADDER, s, b, cols)
    check_grad_rows(out["dB"][cols].double().cpu().numpy(), gB, "dB rows")


def test_clip_n65536_sampled_and_properties(ctx):
    kind, A16, B16, s, b = synth.workload("clip_n65536_hardneg")
    out = run(ctx, kind, A16, B16, s, b)
    check_loss_is_mean_of_terms(out, kind)
    rows = sample(A16.shape[0], 512, 3)
    lse_r, pos_r = oracle.row_stats(kind, A16, B16, LADDER, s, b, rows)
    check_terms(out["row_terms"][:, rows].double().cpu().numpy(), (lse_r - pos_r).T, "row terms")
    cols = sample(B16.shape[0], 512, 4)
    lse_c, pos_c = oracle.row_stats(kind, B16, A16, LADDER, s, b, cols)
    check_terms(out["col_terms"][:, cols].double().cpu().numpy(), (lse_c - pos_c).T, "col terms")
    # gradient rows of both sides against the oracle, from every row's and column's normaliser
    lse_a, _ = oracle.softmax_normalisers(kind, A16, B16, LADDER, s)
    lse_b, _ = oracle.softmax_normalisers(kind, B16, A16, LADDER, s)
    np.testing.assert_allclose(lse_a[:, rows], lse_r.T, rtol=1e-12)  # the two oracle routes agree
    np.testing.assert_allclose(lse_b[:, cols], lse_c.T, rtol=1e-12)
    gA = oracle.grad_rows(kind, True, A16, B16, LADDER, s, b, rows, lse_x=lse_a, lse_y=lse_b)
    check_grad_rows(out["dA"][rows].double().cpu().numpy(), gA, "dA rows")
    gB = oracle.grad_rows(kind, False, B16, A16, LADDER, s, b, cols, lse_x=lse_b, lse_y=lse_a)
    check_grad_rows(out["dB"][cols].double().cpu().numpy(), gB, "dB rows")
    check_euler(A16, out["dA"], "dA")
    check_euler(B16, out["dB"], "dB")
    assert torch.all(out["dA"][:, LADDER[-1]:] == 0) if A16.shape[1] > LADDER[-1] else True
    # swap symmetry: CLIP(B, A) has the same loss and exchanges the gradients
    sw = run(ctx, kind, B16, A16, s, b)
    np.testing.assert_allclose(sw["loss"].cpu().numpy(), out["loss"].cpu().numpy(), rtol=1e-4)
    for g1, g2, what in ((sw["dA"], out["dB"], "dA<->dB"), (sw["dB"], out["dA"], "dB<->dA")):
        err = (g1 - g2).abs().max().item()
        assert err <= 1e-2 * g2.abs().max().item(), what


def test_clip_n65536_at_the_clip_clamp_sampled(ctx):
    """tau = 100 (CLIP's clamp) at the full size: the max-shifted statistics (a max pass, the
    shifts of 65536 rows and columns over 512 row blocks, shifted sums, two exponentials in the
    weight pass).  Noise 6 puts the positives' cosine near 0.16, where the fixed shift would lose
    every sum to fp32 underflow; the loss stays O(1)."""
    kind, s, b = "clip", 100.0, 0.0
    A16, B16 = synth.paired(65536, 1024, 6.0, 31)
    out = run(ctx, kind, A16, B16, s, b)
    check_loss_is_mean_of_terms(out, kind)
    rows = sample(A16.shape[0], 256, 6)
    check_terms(out["row_terms"][:, rows].double().cpu().numpy(),
                oracle.row_terms_sampled(kind, A16, B16, LADDER, s, b, rows), "row terms")
    cols = sample(B16.shape[0], 256, 7)
    check_terms(out["col_terms"][:, cols].double().cpu().numpy(),
                oracle.row_terms_sampled(kind, B16, A16, LADDER, s, b, cols), "col terms")
    check_euler(A16, out["dA"], "dA")
    check_euler(B16, out["dB"], "dB")


def test_clip_n65536_in_two_large_chunks(ctx):
    """A workspace that holds 40960 x 65536 weights cuts the backward into about square chunks
    (2 x 2 here).  Each chunk's dA grid is more than four waves of CTA pairs, so its two
    contractions run as separate launches; dA adds over the chunks of B's rows and dB over the
    chunks of A's rows.  The chunked result matches the one-chunk result up to the fp32
    rounding of adding two chunks (the loss, from the forward, exactly)."""
    kind, A16, B16, s, b = synth.workload("clip_n65536_hardneg")
    N, D = A16.shape
    k = ctx.KINDS[kind]
    wmin = ctx.uf_contrastive_workspace_min(N, N, D, LADDER, k, True)  # the smallest chunk
    ws = torch.empty(wmin + len(LADDER) * (40960 - 128) * N * 2, dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    A, B = dev(A16), dev(B16)
    two = ctx.contrastive_fwd_bwd(A, B, kind, LADDER, s, b, grads=True, workspace=ws, device_status=status)
    del ws
    one = ctx.contrastive_fwd_bwd(A, B, kind, LADDER, s, b, grads=True, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(two["loss"], one["loss"])
    for side in ("dA", "dB"):
        err = (two[side] - one[side]).abs().max().item()
        assert err <= 1e-4 * one[side].abs().max().item(), (side, err)


def test_rows_q8192_k262144_sampled(ctx):
    kind, Q16, K16, s, b = synth.workload("rows_q8192_k262144")
    Nq, Nk = Q16.shape[0], K16.shape[0]
    out = run(ctx, kind, Q16, K16, s, b)
    check_loss_is_mean_of_terms(out, kind)
    assert torch.all(out["col_terms"] == 0)
    rows = sample(Nq, 512, 5)
    lse, pos = oracle.row_stats(kind, Q16, K16, LADDER, s, b, rows)
    check_terms(out["row_terms"][:, rows].double().cpu().numpy(), (lse - pos).T, "query terms")
    # every query's normaliser: the keys' gradient rows sum over all queries
    lse_q, _ = oracle.softmax_normalisers(kind, Q16, K16, LADDER, s)
    np.testing.assert_allclose(lse_q[:, rows], lse.T, rtol=1e-12)  # the two oracle routes agree
    gQ = oracle.grad_rows(kind, True, Q16, K16, LADDER, s, b, rows, lse_x=lse_q)
    check_grad_rows(out["dA"][rows].double().cpu().numpy(), gQ, "query gradient rows")
    # 512 key rows: half among the positives' keys (< Nq), half among the negatives only
    keys = np.concatenate([sample(Nq, 256, 8), Nq + sample(Nk - Nq, 256, 9)])
    gK = oracle.grad_rows(kind, False, K16, Q16, LADDER, s, b, keys, lse_y=lse_q)
    check_grad_rows(out["dB"][keys].double().cpu().numpy(), gK, "key gradient rows")
    check_euler(Q16, out["dA"], "dA")
    check_euler(K16, out["dB"], "dB")


MERGED = [
    # kind, Na, Nb, D, prefixes, scale, bias, noise, seed: long contractions (more than one wave
    # of CTA pairs) with the weights in one chunk, where the two widest prefixes share one weight
    # array below the second widest's end (a multiple of 512); CLIP and ROWS
    ("clip", 6144, 6144, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 41),
    ("rows", 1536, 12288, 1024, LADDER, 1 / 0.05, 0.0, 0.8, 43),
    ("clip", 5120, 5120, 2048, (64, 128, 256, 512, 1024, 2048), 1 / 0.07, 0.0, 1.0, 44),
    ("clip", 5376, 5376, 1024, LADDER, 60.0, 0.0, 2.0, 45),  # the max-shifted statistics
    ("rows", 2048, 10240, 1024, LADDER, 80.0, 0.0, 2.0, 46),  # ROWS on the max-shifted path
    ("clip", 5120, 5120, 1024, (512, 1024), 1 / 0.07, 0.0, 1.0, 47),  # two prefixes: nothing below the merge
    ("clip", 2560, 2560, 4096, (64, 256, 1024, 4096), 1 / 0.07, 0.0, 1.0, 48),  # six slice groups above it
]


@pytest.mark.parametrize("kind,Na,Nb,D,pre,scale,bias,noise,seed", MERGED)
def test_merged_widest_prefixes_sampled(ctx, kind, Na, Nb, D, pre, scale, bias, noise, seed):
    """The merged path (it reduces prefix n-1's partial row scalars in a second launch of the
    norm-backward group) against the oracle's gradient rows, and the Euler identity, whose
    projection scalars the merge recovers as (x . G of both prefixes) - (prefix n-1's)."""
    A16, B16 = (synth.queries_keys(Na, Nb, D, noise, seed) if kind == "rows" else synth.paired(Na, D, noise, seed))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ctx.uf_contrastive_profile(True)
    out = ctx.contrastive_fwd_bwd(dev(A16), dev(B16), kind, pre, scale, bias, grads=True, terms=True,
                                  device_status=status)
    torch.cuda.synchronize()
    launches = ctx.uf_contrastive_profile_read(ctx.KERNEL_GROUPS.index("norm_bwd"))[2]
    ctx.uf_contrastive_profile(False)
    assert int(status.item()) == 0
    assert launches == 2, "the merged path did not run (its partial sums are reduced in a second launch)"
    rows = sample(Na, 128, seed)
    cols = sample(Nb, 128, seed + 100)
    lse_a = lse_b = None
    if kind != "siglip":
        lse_a, _ = oracle.softmax_normalisers(kind, A16, B16, pre, scale)
        if kind == "clip":
            lse_b, _ = oracle.softmax_normalisers(kind, B16, A16, pre, scale)
    if kind == "rows":
        gA = oracle.grad_rows(kind, True, A16, B16, pre, scale, bias, rows, lse_x=lse_a)
        gB = oracle.grad_rows(kind, False, B16, A16, pre, scale, bias, cols, lse_y=lse_a)
    else:
        gA = oracle.grad_rows(kind, True, A16, B16, pre, scale, bias, rows, lse_x=lse_a, lse_y=lse_b)
        gB = oracle.grad_rows(kind, False, B16, A16, pre, scale, bias, cols, lse_x=lse_b, lse_y=lse_a)
    check_grad_rows(out["dA"][rows].double().cpu().numpy(), gA, "dA rows")
    check_grad_rows(out["dB"][cols].double().cpu().numpy(), gB, "dB rows")
    check_euler(A16, out["dA"], "dA")
    check_euler(B16, out["dB"], "dB")
