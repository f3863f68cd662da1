"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Tolerances (the acceptance bar of the Matryoshka loss build): per-prefix loss relative
error <= 2e-3; gradient max-abs error <= 1e-2 * max|grad|.  Per-row terms are held to
2e-3 of the largest term.
"""
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


def run(binding, kind, A16, B16, pre, scale, bias, weights=None, grads=True, workspace=None, scale_grads=False):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = binding.contrastive_fwd_bwd(dev(A16), dev(B16), kind, pre, scale, bias, weights, grads=grads, terms=True,
                                      workspace=workspace, device_status=status, scale_grads=scale_grads)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, "a kernel reported a timeout"
    return {k: v.double().cpu().numpy() for k, v in out.items()}


def check_loss(got, ref, scale=1.0):
    # the oracle's InfoNCE loss is LSE - s_ii, a difference of O(scale) float64 numbers: below
    # about 64 ulp(scale) it is rounding (a batch of one pair gives +-1e-15 for an exact 0)
    floor = 64 * np.finfo(np.float64).eps * max(abs(scale), 1.0)
    err = np.abs(got - ref)
    assert np.all(err <= LOSS_RTOL * np.abs(ref) + floor), f"loss {got} vs oracle {ref}"


def check_grad(got, ref, what):
    err = np.abs(got - ref).max()
    scale = np.abs(ref).max()
    # (+1e-12: the oracle's float64 rounding where the gradient vanishes exactly, e.g. one pair)
    assert err <= GRAD_FRAC * scale + 1e-12, f"{what}: max-abs err {err:.3e} > {GRAD_FRAC} * {scale:.3e}"


def check_terms(got, ref, what, scale=1.0):
    err = np.abs(got - ref).max()
    floor = 64 * np.finfo(np.float64).eps * max(abs(scale), 1.0)  # as in check_loss
    assert err <= LOSS_RTOL * np.abs(ref).max() + floor, f"{what}: err {err:.3e}"


def make(kind, Na, Nb, D, seed, noise):
    if kind == "rows":
        return synth.queries_keys(Na, Nb, D, noise, seed)
    return synth.paired(Na, D, noise, seed)


SMALL = [
    # kind, Na, Nb, D, prefixes, scale, bias, noise, seed
    ("clip", 256, 256, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 0),     # the N=256 benchmark configuration itself
    ("clip", 300, 300, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 11),    # ragged tail (300 = 2*128 + 44)
    ("clip", 640, 640, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 12),    # five tiles per row
    ("siglip", 300, 300, 1024, LADDER, 10.0, -10.0, 0.7, 13),
    ("siglip", 512, 512, 1024, LADDER, 10.0, -10.0, 0.7, 14),
    ("rows", 200, 700, 1024, LADDER, 1 / 0.05, 0.0, 0.8, 15),     # ragged queries and keys
    ("clip", 257, 257, 384, (64, 192, 384), 5.0, 0.0, 1.0, 16),   # another ladder; partial gradient slice
    ("clip", 130, 130, 1024, (1024,), 1 / 0.07, 0.0, 1.0, 17),    # one prefix
    ("siglip", 200, 200, 640, (128, 320, 512), 4.0, -2.0, 0.7, 18),  # last prefix < D: zero tail columns
    ("rows", 1, 300, 1024, LADDER, 1 / 0.05, 0.0, 0.8, 19),       # one query
    ("clip", 192, 192, 1024, LADDER, 40.0, 0.0, 3.0, 21),         # the largest supported tau
    ("clip", 260, 260, 640, (64, 320, 640), 5.0, 0.0, 1.0, 22),   # an odd number of 256-dimension slices
    # one pair: CLIP has no negative (every row term is exactly 0), SigLIP one cell
    ("clip", 1, 1, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 28),
    ("siglip", 1, 1, 1024, LADDER, 10.0, -10.0, 0.7, 29),
    # the limits of the API: one 64-wide band, eight prefixes, D up to 4096 (sixteen slices)
    ("clip", 300, 300, 64, (64,), 1 / 0.07, 0.0, 1.0, 23),
    ("clip", 260, 260, 512, (64, 128, 192, 256, 320, 384, 448, 512), 1 / 0.07, 0.0, 1.0, 24),
    ("siglip", 200, 200, 2048, (64, 128, 256, 512, 1024, 2048), 10.0, -10.0, 0.7, 25),
    ("rows", 130, 400, 4096, (64, 256, 1024, 4096), 1 / 0.05, 0.0, 0.8, 26),
    ("clip", 256, 256, 4096, (64, 128, 256, 512, 1024, 2048, 4096), 1 / 0.07, 0.0, 1.0, 27),
]


@pytest.mark.parametrize("kind,Na,Nb,D,pre,scale,bias,noise,seed", SMALL)
def test_parity_small(ctx, kind, Na, Nb, D, pre, scale, bias, noise, seed):
    A16, B16 = make(kind, Na, Nb, D, seed, noise)
    w = np.linspace(0.5, 1.5, len(pre))
    got = run(ctx, kind, A16, B16, pre, scale, bias, weights=list(w))
    ref = oracle.fwd_bwd(kind, A16, B16, pre, scale, bias, w)
    check_loss(got["loss"], ref["loss"], scale)
    check_terms(got["row_terms"], ref["row_terms"], "row terms", scale)
    if kind == "clip":
        check_terms(got["col_terms"], ref["col_terms"], "col terms", scale)
    else:  # the library defines column terms for CLIP only and writes 0 otherwise
        assert np.all(got["col_terms"] == 0)
    check_grad(got["dA"], ref["dA"], "dA")
    check_grad(got["dB"], ref["dB"], "dB")
    assert np.all(got["dA"][:, pre[-1]:] == 0) and np.all(got["dB"][:, pre[-1]:] == 0)


CHUNKED = [
    # kind, Na, Nb, D, prefixes, scale, bias, noise, seed: the smallest workspace, so the
    # backward weights are cut into 128 x 256 chunks (dA adds over column chunks, dB over row chunks)
    ("clip", 640, 640, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 51),
    ("siglip", 300, 300, 1024, LADDER, 10.0, -10.0, 0.7, 52),
    ("rows", 200, 700, 1024, LADDER, 1 / 0.05, 0.0, 0.8, 53),
    ("clip", 257, 257, 384, (64, 192, 384), 5.0, 0.0, 1.0, 54),
]


@pytest.mark.parametrize("kind,Na,Nb,D,pre,scale,bias,noise,seed", CHUNKED)
def test_parity_smallest_workspace(ctx, kind, Na, Nb, D, pre, scale, bias, noise, seed):
    A16, B16 = make(kind, Na, Nb, D, seed, noise)
    k = ctx.KINDS[kind]
    wmin = ctx.uf_contrastive_workspace_min(Na, Nb, D, pre, k, True)
    assert wmin < ctx.uf_contrastive_workspace_size(Na, Nb, D, pre, k, True)  # more than one chunk
    ws = torch.empty(wmin, dtype=torch.uint8, device="cuda")
    got = run(ctx, kind, A16, B16, pre, scale, bias, workspace=ws)
    ref = oracle.fwd_bwd(kind, A16, B16, pre, scale, bias)
    check_loss(got["loss"], ref["loss"])
    check_grad(got["dA"], ref["dA"], "dA")
    check_grad(got["dB"], ref["dB"], "dB")
    full = run(ctx, kind, A16, B16, pre, scale, bias)  # one chunk: the same loss bits
    assert np.array_equal(got["loss"], full["loss"])


def test_forward_only_matches(ctx):
    A16, B16 = make("clip", 300, 300, 1024, 31, 1.0)
    full = run(ctx, "clip", A16, B16, LADDER, 1 / 0.07, 0.0)
    fwd = run(ctx, "clip", A16, B16, LADDER, 1 / 0.07, 0.0, grads=False)
    assert np.array_equal(full["loss"], fwd["loss"])
    S16, T16 = make("siglip", 300, 300, 1024, 32, 0.7)
    ref = oracle.fwd_bwd("siglip", S16, T16, LADDER, 10.0, -10.0, grads=False)
    check_loss(run(ctx, "siglip", S16, T16, LADDER, 10.0, -10.0, grads=False)["loss"], ref["loss"])


def test_identical_embeddings_give_ln_n(ctx):
    v = np.random.default_rng(0).standard_normal(1024)
    A16 = synth.round_to_bf16_bits(np.tile(v, (384, 1)))
    got = run(ctx, "clip", A16, A16, LADDER, 1 / 0.07, 0.0)
    np.testing.assert_allclose(got["loss"], np.log(384), rtol=LOSS_RTOL)
    scale = np.abs(run(ctx, "clip", *make("clip", 384, 384, 1024, 3, 1.0), LADDER, 1 / 0.07, 0.0)["dA"]).max()
    assert np.abs(got["dA"]).max() <= GRAD_FRAC * scale


def test_single_pair(ctx):
    """N = 1: the only logit is the positive, so L = 0 and every gradient vanishes."""
    A16, B16 = make("clip", 1, 1, 128, 20, 1.0)
    got = run(ctx, "clip", A16, B16, (64, 128), 1 / 0.07, 0.0)
    assert np.abs(got["loss"]).max() < 1e-5
    assert np.abs(got["dA"]).max() < 1e-6 and np.abs(got["dB"]).max() < 1e-6


def test_deterministic(ctx):
    A16, B16 = make("clip", 640, 640, 1024, 40, 1.0)
    r1 = run(ctx, "clip", A16, B16, LADDER, 1 / 0.07, 0.0)
    r2 = run(ctx, "clip", A16, B16, LADDER, 1 / 0.07, 0.0)
    for k in r1:
        assert np.array_equal(r1[k], r2[k]), k


def logit_grad_l1(kind, A16, B16, pre, scale, bias, w):
    """(sum_k w_k sum_ij |dL_k/dx_ij| |cos_ij|, sum_k w_k sum_ij |dL_k/dx_ij|), x the logits.

    Only a tolerance: both gradients are sums over the score matrix of dL/dx_ij times cos_ij
    (logit scale) or times 1 (bias), and the library rounds every dL/dcos_ij to bf16
    (relative error <= 2^-9) before it sums them, so the error of each sum is at most
    2^-9 times the matching sum of magnitudes."""
    A, B = synth.bf16_bits_to_float(A16), synth.bf16_bits_to_float(B16)
    Na = A.shape[0]
    m_cos = m_one = 0.0
    for k, p in enumerate(pre):
        a = A[:, :p] / np.linalg.norm(A[:, :p], axis=1, keepdims=True)
        b = B[:, :p] / np.linalg.norm(B[:, :p], axis=1, keepdims=True)
        cos = a @ b.T
        x = scale * cos + (bias if kind == "siglip" else 0.0)
        eye = np.zeros_like(x)
        eye[np.arange(min(x.shape)), np.arange(min(x.shape))] = 1.0
        if kind == "siglip":
            g = (1.0 / (1.0 + np.exp(-x)) - eye) / Na
        else:
            pr = np.exp(x - x.max(1, keepdims=True))
            g = (pr / pr.sum(1, keepdims=True) - eye) / Na
            if kind == "clip":
                pc = np.exp(x - x.max(0, keepdims=True))
                g = 0.5 * (g + (pc / pc.sum(0, keepdims=True) - eye) / Na)
        m_cos += w[k] * np.sum(np.abs(g) * np.abs(cos))
        m_one += w[k] * np.sum(np.abs(g))
    return m_cos, m_one


SCALE_GRADS = [
    # kind, Na, Nb, D, prefixes, scale, bias, noise, seed, smallest workspace
    ("clip", 300, 300, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 71, False),
    ("clip", 640, 640, 1024, LADDER, 1 / 0.07, 0.0, 1.0, 72, True),
    ("clip", 257, 257, 384, (64, 192, 384), 40.0, 0.0, 3.0, 73, False),
    ("siglip", 300, 300, 1024, LADDER, 10.0, -10.0, 0.7, 74, False),
    ("siglip", 512, 512, 1024, LADDER, 4.0, -2.0, 0.7, 75, True),     # many negatives with sizeable sigmoid
    ("siglip", 200, 200, 640, (128, 320, 512), 4.0, 1.0, 0.7, 76, False),
    ("rows", 200, 700, 1024, LADDER, 1 / 0.05, 0.0, 0.8, 77, False),
    ("rows", 1, 300, 1024, LADDER, 1 / 0.05, 0.0, 0.8, 78, False),
]


@pytest.mark.parametrize("kind,Na,Nb,D,pre,scale,bias,noise,seed,small_ws", SCALE_GRADS)
def test_parity_scale_and_bias_gradients(ctx, kind, Na, Nb, D, pre, scale, bias, noise, seed, small_ws):
    A16, B16 = make(kind, Na, Nb, D, seed, noise)
    w = list(np.linspace(1.5, 0.5, len(pre)))
    ws = None
    if small_ws:
        wmin = ctx.uf_contrastive_workspace_min(Na, Nb, D, pre, ctx.KINDS[kind], True)
        ws = torch.empty(wmin, dtype=torch.uint8, device="cuda")
    got = run(ctx, kind, A16, B16, pre, scale, bias, weights=w, workspace=ws, scale_grads=True)
    ds, db = oracle.scale_grads(kind, A16, B16, pre, scale, bias, w)
    m_cos, m_one = logit_grad_l1(kind, A16, B16, pre, scale, bias, w)
    tol_s = 2.0 ** -8 * m_cos + 1e-5 * abs(ds)   # twice the bf16 rounding bound, plus fp32 sums
    tol_b = 2.0 ** -8 * m_one + 1e-5 * abs(db)
    assert abs(got["d_logit_scale"][0] - ds) <= tol_s, f"dL/dscale {got['d_logit_scale'][0]} vs oracle {ds}"
    if kind == "siglip":
        assert abs(got["d_bias"][0] - db) <= tol_b, f"dL/dbias {got['d_bias'][0]} vs oracle {db}"
    else:
        assert got["d_bias"][0] == 0.0
    # asking for them changes nothing else
    plain = run(ctx, kind, A16, B16, pre, scale, bias, weights=w, workspace=ws)
    for key in ("loss", "dA", "dB", "row_terms"):
        assert np.array_equal(got[key], plain[key]), key
