"""Run a few calls of the loss on one synthetic batch (for profilers such as ncu).

  python -m contrastive_embedding_loss_gb300.profile_call --kind clip --n 32768 --warmup 1 --calls 1

Each call is one full uf_contrastive_fwd_bwd (forward, loss, backward).  The kernel
launch order per CLIP call (tau <= 40, one weight chunk) is: prep, transpose (both sides),
fwd_kernel, stats, wgt_kernel, gemm_kernel (dA, K-major weights), gemm_kernel (dB, MN-major
weights) or, below four waves of CTA pairs, gemm_kernel_both (both), norm_bwd (both sides).
"""
import argparse

import numpy as np


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--kind", default="clip", choices=["clip", "siglip", "rows"])
    ap.add_argument("--n", type=int, default=32768, help="pairs (queries for rows)")
    ap.add_argument("--nk", type=int, default=0, help="keys for rows (default 8 * n)")
    ap.add_argument("--d", type=int, default=1024)
    ap.add_argument("--warmup", type=int, default=1)
    ap.add_argument("--calls", type=int, default=1)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--weights-gib", type=float, default=0.0,
                    help="cap the backward weight array at this many GiB (chunked weights; 0: the default)")
    a = ap.parse_args()

    import torch

    from . import binding, synth

    pre = tuple(p for p in (64, 128, 256, 512, 1024, 2048, 4096) if p <= a.d)
    if a.kind == "rows":
        A16, B16 = synth.queries_keys(a.n, a.nk or 8 * a.n, a.d, 0.8, a.seed)
        scale, bias = 1 / 0.05, 0.0
    else:
        A16, B16 = synth.paired(a.n, a.d, 0.7 if a.kind == "siglip" else 1.0, a.seed)
        scale, bias = (10.0, -10.0) if a.kind == "siglip" else (1 / 0.07, 0.0)
    dev = torch.device("cuda:0")
    A = torch.from_numpy(A16.view(np.int16)).view(torch.bfloat16).to(dev)
    B = torch.from_numpy(B16.view(np.int16)).view(torch.bfloat16).to(dev)
    assert binding.uf_contrastive_init(0) == binding.UF_OK
    args = (A.shape[0], B.shape[0], a.d, pre, binding.KINDS[a.kind], 1)
    nbytes = binding.uf_contrastive_workspace_size(*args)
    if a.weights_gib > 0:
        nbytes = min(nbytes, binding.uf_contrastive_workspace_min(*args) + int(a.weights_gib * (1 << 30)))
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    out = None
    for _ in range(a.warmup + a.calls):
        out = binding.contrastive_fwd_bwd(A, B, a.kind, pre, scale, bias, workspace=ws)
    torch.cuda.synchronize()
    print("loss per prefix:", out["loss"].cpu().numpy().tolist())


if __name__ == "__main__":
    main()
