"""uf_contrastive_fwd_bwd_static: the loss for callers that cannot allocate device memory.

Such callers (hosts that reserve all memory at start-up, plugins whose application owns
every device buffer, fixed-pool allocators) cannot pass a workspace, so the library
keeps one fixed-size scratch array per GPU.  These tests call that entry point through
the C ABI twice in a row and hold each result to the tolerances of the parity tests
against the ordinary (caller-workspace) entry point on the same inputs.  This file is
collected last so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest

from contrastive_embedding_loss_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LADDER = (64, 128, 256, 512, 1024)


@pytest.fixture(scope="module")
def binding():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding as b

    assert b.uf_contrastive_init(0) == 0
    return b


def _dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _static_call(b, kind, A, B, scale, bias, grads):
    Na, D = A.shape
    Nb = B.shape[0]
    n = len(LADDER)
    out = {"loss": torch.full((n,), float("nan"), device="cuda"),
           "row_terms": torch.full((n, Na), float("nan"), device="cuda"),
           "col_terms": torch.full((n, Nb), float("nan"), device="cuda")}
    if grads:
        out["dA"] = torch.full((Na, D), float("nan"), device="cuda")
        out["dB"] = torch.full((Nb, D), float("nan"), device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    st = b.uf_contrastive_fwd_bwd_static(A.data_ptr(), B.data_ptr(), Na, Nb, D, LADDER, b.KINDS[kind], scale, bias,
                                         None, out["loss"].data_ptr(), out["row_terms"].data_ptr(),
                                         out["col_terms"].data_ptr(), ptr(out.get("dA")), ptr(out.get("dB")),
                                         status.data_ptr(), torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert st == 0, b.uf_status_name(st)
    assert int(status.item()) == 0
    return out


CASES = [
    ("clip", 4096, 4096, 1 / 0.07, 0.0, True),    # the backward weights take several chunks
    ("siglip", 700, 700, 10.0, -10.0, True),      # ragged tiles
    ("rows", 300, 9000, 1 / 0.05, 0.0, False),    # forward only
]


@pytest.mark.parametrize("kind,Na,Nb,scale,bias,grads", CASES)
def test_static_entry_matches_workspace_entry(binding, kind, Na, Nb, scale, bias, grads):
    if kind == "rows":
        A16, B16 = synth.queries_keys(Na, Nb, 1024, 0.8, 7)
    else:
        A16, B16 = synth.paired(Na, 1024, 0.7 if kind == "siglip" else 1.0, 7)
    A, B = _dev(A16), _dev(B16)
    ref = binding.contrastive_fwd_bwd(A, B, kind, LADDER, scale, bias, grads=grads, terms=True)
    torch.cuda.synchronize()
    for _ in range(2):  # two calls in a row share (and reuse) the one scratch array
        got = _static_call(binding, kind, A, B, scale, bias, grads)
        rel = ((got["loss"] - ref["loss"]).abs() / ref["loss"].abs()).max().item()
        assert rel <= 2e-3
        for key in ("row_terms", "col_terms"):
            err = (got[key] - ref[key]).abs().max().item()
            assert err <= 2e-3 * max(ref[key].abs().max().item(), 1e-30), key
        if grads:
            for key in ("dA", "dB"):
                err = (got[key] - ref[key]).abs().max().item()
                assert err <= 1e-2 * ref[key].abs().max().item(), key


def test_static_entry_rejects_batches_beyond_its_scratch(binding):
    N = 16384
    A16, B16 = synth.paired(N, 1024, 1.0, 8)
    need = binding.uf_contrastive_workspace_min(N, N, 1024, LADDER, 0, True)
    assert need > binding.UF_STATIC_WORKSPACE_BYTES
    A, B = _dev(A16), _dev(B16)
    loss = torch.zeros(len(LADDER), device="cuda")
    dA = torch.zeros((N, 1024), device="cuda")
    dB = torch.zeros((N, 1024), device="cuda")
    st = binding.uf_contrastive_fwd_bwd_static(A.data_ptr(), B.data_ptr(), N, N, 1024, LADDER, 0, 1 / 0.07, 0.0,
                                               None, loss.data_ptr(), None, None, dA.data_ptr(), dB.data_ptr(), None,
                                               torch.cuda.current_stream().cuda_stream)
    assert binding.uf_status_name(st) == "workspace-too-small"
    torch.cuda.synchronize()
    assert torch.all(loss == 0)  # nothing was enqueued
