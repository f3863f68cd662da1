"""Memory safety without a sanitizer: every buffer the library may write sits inside a larger
allocation filled with a canary pattern, in front of it and behind it.  After the call, each
canary region must be unchanged.  The buffers are the workspace, the loss, the row and column
terms, dA and dB.  The cases are CLIP, SigLIP, ROWS and CLIP with the smallest workspace (the
backward in weight chunks), at ragged sizes."""
import numpy as np
import pytest

from contrastive_embedding_loss_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LADDER = (64, 128, 256, 512, 1024)
PAD = 4096  # bytes of canary on each side (keeps 256-byte alignment)
CANARY = 0xA5


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding

    assert binding.uf_contrastive_init(0) == 0
    return binding


class Guarded:
    """nbytes of device memory with PAD canary bytes before and after it."""

    def __init__(self, nbytes):
        self.nbytes = int(nbytes)
        self.raw = torch.full((PAD + self.nbytes + PAD,), CANARY, dtype=torch.uint8, device="cuda")

    @property
    def ptr(self):
        return self.raw.data_ptr() + PAD

    def intact(self):
        front = self.raw[:PAD]
        back = self.raw[PAD + self.nbytes:]
        return bool((front == CANARY).all()) and bool((back == CANARY).all())


@pytest.mark.parametrize("kind,Na,Nb,smallest_ws", [
    ("clip", 1000, 1000, False),
    ("clip", 1000, 1000, True),
    ("siglip", 777, 777, False),
    ("rows", 300, 1300, False),
])
def test_no_write_outside_the_buffers(ctx, kind, Na, Nb, smallest_ws):
    binding = ctx
    D = 1024
    if kind == "rows":
        A16, B16 = synth.queries_keys(Na, Nb, D, 1.0, 21)
    else:
        A16, B16 = synth.paired(Na, D, 1.0, 22)
    dev = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    A, B = dev(A16), dev(B16)
    k = binding.KINDS[kind]
    n = len(LADDER)
    size = binding.uf_contrastive_workspace_min if smallest_ws else binding.uf_contrastive_workspace_size
    ws_bytes = size(Na, Nb, D, LADDER, k, True)
    bufs = {
        "workspace": Guarded(ws_bytes),
        "loss": Guarded(n * 4),
        "row_terms": Guarded(n * Na * 4),
        "col_terms": Guarded(n * Nb * 4),
        "dA": Guarded(Na * D * 4),
        "dB": Guarded(Nb * D * 4),
    }
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    scale, bias = (10.0, -10.0) if kind == "siglip" else (1 / 0.07, 0.0)
    st = binding.uf_contrastive_fwd_bwd(A.data_ptr(), B.data_ptr(), Na, Nb, D, LADDER, k, scale, bias, None,
                                        bufs["loss"].ptr, bufs["row_terms"].ptr, bufs["col_terms"].ptr,
                                        bufs["dA"].ptr, bufs["dB"].ptr, bufs["workspace"].ptr, ws_bytes,
                                        status.data_ptr(), stream.cuda_stream)
    torch.cuda.synchronize()
    assert st == 0 and int(status.item()) == 0
    for name, g in bufs.items():
        assert g.intact(), f"{name}: a canary byte changed"
    # the outputs were written (no canary pattern left inside them) and are finite
    loss = bufs["loss"].raw[PAD:PAD + n * 4].view(torch.float32)
    dA = bufs["dA"].raw[PAD:PAD + Na * D * 4].view(torch.float32)
    assert torch.isfinite(loss).all() and torch.isfinite(dA).all()
    ref = binding.contrastive_fwd_bwd(A, B, kind, LADDER, scale, bias, grads=True)
    torch.cuda.synchronize()
    np.testing.assert_allclose(loss.cpu().numpy(), ref["loss"].cpu().numpy(), rtol=1e-5)
