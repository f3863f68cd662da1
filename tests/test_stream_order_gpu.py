"""Back-to-back calls on one stream, with no synchronisation between them.

Every kernel of the library is launched with programmatic dependent launch: it may be scheduled
while the kernel before it on the stream drains, and it waits for that grid (griddepcontrol.wait)
before it touches memory.  These tests queue several calls, of different kinds and sizes, with a
PyTorch kernel rewriting an input between two of them, and check each result against the same
call run alone and synchronised: bit-identical, since every pass reduces in a fixed order.  A
call that read an input before the kernel writing it had finished, or a kernel that read the
statistics of a call still in flight, would differ.
"""
import numpy as np
import pytest

from contrastive_embedding_loss_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

LADDER = (64, 128, 256, 512, 1024)


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding

    assert binding.uf_contrastive_init(0) == 0
    return binding


def dev(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


class Call:
    """One call's inputs, outputs and workspace, all preallocated, so that queueing it only
    launches kernels."""

    def __init__(self, lib, kind, n, seed, scale, bias):
        self.lib, self.kind, self.scale, self.bias = lib, kind, scale, bias
        A16, B16 = synth.paired(n, 1024, 0.7 if kind == "siglip" else 1.0, seed)
        self.A, self.B = dev(A16), dev(B16)
        k = lib.KINDS[kind]
        self.k = k
        self.ws_bytes = lib.uf_contrastive_workspace_size(n, n, 1024, LADDER, k, True)
        self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device="cuda")
        self.loss = torch.empty(len(LADDER), dtype=torch.float32, device="cuda")
        self.dA = torch.empty((n, 1024), dtype=torch.float32, device="cuda")
        self.dB = torch.empty((n, 1024), dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.n = n

    def queue(self):
        st = self.lib.uf_contrastive_fwd_bwd(self.A.data_ptr(), self.B.data_ptr(), self.n, self.n, 1024, LADDER,
                                             self.k, self.scale, self.bias, None, self.loss.data_ptr(), None, None,
                                             self.dA.data_ptr(), self.dB.data_ptr(), self.ws.data_ptr(),
                                             self.ws_bytes, self.status.data_ptr(),
                                             torch.cuda.current_stream().cuda_stream)
        assert st == self.lib.UF_OK

    def result(self):
        return [t.clone() for t in (self.loss, self.dA, self.dB)]


def alone(call):
    torch.cuda.synchronize()
    call.queue()
    torch.cuda.synchronize()
    assert int(call.status.item()) == 0
    return call.result()


def same(a, b):
    return all(torch.equal(x, y) for x, y in zip(a, b))


def test_back_to_back_calls_match_synchronised_ones(lib):
    calls = [Call(lib, "clip", 4096, 61, 1 / 0.07, 0.0), Call(lib, "clip", 256, 62, 1 / 0.07, 0.0),
             Call(lib, "siglip", 1000, 63, 10.0, -10.0), Call(lib, "clip", 8192, 64, 1 / 0.07, 0.0)]
    ref = [alone(c) for c in calls]
    torch.cuda.synchronize()
    order = [0, 1, 2, 3, 0, 3, 1, 2]
    got = {}
    for i in order:  # one stream, no synchronisation in between
        calls[i].queue()
        got.setdefault(i, []).append(calls[i].result())  # clone kernels queued between the calls
    torch.cuda.synchronize()
    for c in calls:
        assert int(c.status.item()) == 0
    for i, results in got.items():
        for r in results:
            assert same(r, ref[i]), f"call {i} differs when queued back to back"


def test_input_rewritten_between_calls(lib):
    """A PyTorch kernel scales A between two queued calls: the second call must see the new A,
    the first the old one, and each must equal the synchronised call on the same values."""
    c = Call(lib, "clip", 4096, 65, 1 / 0.07, 0.0)
    ref_old = alone(c)
    A_old = c.A.clone()
    c.A.mul_(-1.0)  # (exact in bf16: the loss sees the sign-flipped A)
    ref_new = alone(c)
    c.A.copy_(A_old)
    torch.cuda.synchronize()
    c.queue()
    first = c.result()
    c.A.mul_(-1.0)
    c.queue()
    second = c.result()
    torch.cuda.synchronize()
    assert int(c.status.item()) == 0
    assert same(first, ref_old)
    assert same(second, ref_new)
    assert not same(ref_old, ref_new)
