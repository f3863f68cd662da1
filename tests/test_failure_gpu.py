"""The kernels' failure path on the GPU, without a fault: a bounded wait that runs out reports
UF_DEVICE_TIMEOUT in the caller's device status and the context stays usable."""
import time

import numpy as np
import pytest

import oracle
from contrastive_embedding_loss_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from contrastive_embedding_loss_gb300 import binding

    assert binding.uf_contrastive_init(0) == 0
    return binding


def test_bounded_wait_runs_out_and_reports(ctx):
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    t0 = time.perf_counter()
    assert ctx.uf_contrastive_selftest_wait(status.data_ptr(), 200, stream.cuda_stream) == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == 5  # UF_DEVICE_TIMEOUT
    assert 0.15 < dt < 5.0          # it gave up after about its limit, not never and not at once
    # the context is still usable: a loss call right after it is correct
    A16, B16 = synth.paired(256, 1024, 1.0, 41)
    dev = lambda x: torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).cuda()  # noqa: E731
    ok = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = ctx.contrastive_fwd_bwd(dev(A16), dev(B16), "clip", (64, 128, 256, 512, 1024), 1 / 0.07, 0.0,
                                  device_status=ok)
    torch.cuda.synchronize()
    assert int(ok.item()) == 0
    ref = oracle.fwd_bwd("clip", A16, B16, (64, 128, 256, 512, 1024), 1 / 0.07, 0.0)
    np.testing.assert_allclose(out["loss"].cpu().numpy(), ref["loss"], rtol=2e-3)
