"""Benchmark: Matryoshka contrastive loss forward+backward on one GB300 (or N replicas).

A step is one call of uf_contrastive_fwd_bwd over one batch: inverse norms, forward row
statistics, loss, backward score recompute + gradient GEMMs, projection -- every step of
the path.  Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

--impl reference times the float64 CPU oracle on the host cores instead: the pages publish no
runnable implementation of this path, so the oracle stands in as the reference arm.
"""
import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "fwd+bwd pairs/s at 5 prefixes (N=65536, D=1024 bf16); TFLOP/s vs bf16 peak"
LADDER = (64, 128, 256, 512, 1024)
DEFAULT_WORKLOAD = "clip_n65536_hardneg"
ORACLE_SAMPLE_PAIRS = 8192      # cpu_baseline: oracle on the first 8192 pairs (about 10-30 s on 16 cores)
REFERENCE_STEP_PAIRS = 1024     # --impl reference: oracle on the first 1024 pairs per step
COPY_SPLIT = 4                  # end-to-end timing: input copies split over this many streams


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-workspace", action="store_true",
                    help="run with uf_contrastive_workspace_min bytes (the backward in its smallest weight chunks)")
    ap.add_argument("--weights-gib", type=float, default=None,
                    help="run with uf_contrastive_workspace_min bytes plus this many GiB for the weight chunks")
    return ap.parse_args()


def pairs_of(w, A16):
    return A16.shape[0]  # CLIP/SigLIP: N pairs; ROWS: Nq queries


def credited_flops(kind, Na, Nb, D):
    # forward S + backward S + dA + dB for InfoNCE (S is needed twice); SigLIP skips the forward
    return (6 if kind == "siglip" else 8) * Na * Nb * D


def executed_flops(kind, Na, Nb, D, prefixes=None, merged=False):
    """Tensor-core flops the library runs per step: the forward score pass (not for SigLIP,
    whose loss comes out of the weight pass), the weight pass, and the two prefix-expanded
    gradient GEMMs (prefix k contributes p_k dimensions; merged: prefix n-1 none below p_{n-2})."""
    pre = list(prefixes) if prefixes else [D]
    score = 2.0 * Na * Nb * pre[-1]
    gemms = group_flops_executed("gemm", kind, Na, Nb, D, pre, merged)
    return (0.0 if kind == "siglip" else score) + score + gemms


def group_flops(group, kind, Na, Nb, D, prefixes):
    """Algorithmic tensor flops of one kernel group per step (None: not a tensor kernel): the
    method's own work.  A score pass is 2 Na Nb p_n (the prefixes nest, so one K sweep serves
    all of them); each gradient contraction is 2 Na Nb p_n as well (every output dimension d
    receives the running sum of the weights of the prefixes that reach d, so it is contracted
    once)."""
    pre = list(prefixes)
    if group in ("fwd_tile", "bwd_tile"):
        return 2.0 * Na * Nb * pre[-1]
    if group == "gemm":
        return 2 * 2.0 * Na * Nb * pre[-1]  # the dA and the dB contraction
    return None


def group_flops_executed(group, kind, Na, Nb, D, prefixes, merged=False):
    """Tensor flops the library's kernels of one group actually issue per step.  merged: the two
    widest prefixes' weights shared one array below p_{n-2}, so prefix n-1 ran only above it."""
    pre = list(prefixes)
    if group == "gemm":
        dims = sum(pre) - (pre[-2] if merged and len(pre) >= 2 else 0)
        return 2 * 2.0 * Na * Nb * dims  # prefix-expanded: prefix k contributes its p_k dimensions
    return group_flops(group, kind, Na, Nb, D, prefixes)


def group_bytes(group, kind, Na, Nb, D, prefixes):
    """Algorithmic HBM bytes of one kernel group per step: what the method must move for it
    at the least (the two gradient contractions: each writes its fp32 gradient once and reads
    the other side's bf16 embeddings once; the weights never need to leave the chip)."""
    if group == "gemm":
        return 4.0 * (Na + Nb) * D + 2.0 * (Na + Nb) * D
    return None


def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def sub_batch(kind, A16, B16, n):
    # the first n pairs (for ROWS: the first n queries and their n positive keys)
    return A16[:n], B16[:n]


L2_BYTES = 129 * 10**6  # GB300's L2


def l2_policy(A16, B16):
    """How the timed steps stand to L2: the inputs are not flushed between steps, which keeps the
    timing clean only when they are larger than L2 (the benchmark workload: 268 MB)."""
    in_bytes = (A16.shape[0] + B16.shape[0]) * A16.shape[1] * 2
    if in_bytes > L2_BYTES:
        return "inputs larger than L2 (no flush)"
    return f"inputs ({in_bytes / 1e6:.0f} MB) fit in L2 and are not flushed between steps"


def run_config(args, kind, A16, B16, scale, bias, world):
    """The workload as both arms report it (the same dict, so that their lines compare)."""
    return {"workload": args.workload, "kind": kind, "Na": int(A16.shape[0]), "Nb": int(B16.shape[0]),
            "D": int(A16.shape[1]), "prefixes": list(LADDER), "logit_scale": scale, "bias": bias,
            "l2": l2_policy(A16, B16), "parallelism": f"replicas x{world}"}


def oracle_rate(kind, A16, B16, scale, bias, n_sample):
    """Time the oracle on a sub-batch and scale its time to the full batch by cells (N^2)."""
    import oracle

    a, b = sub_batch(kind, A16, B16, n_sample)
    t0 = time.perf_counter()
    oracle.fwd_bwd(kind, a, b, LADDER, scale, bias)
    dt = time.perf_counter() - t0
    full_cells = A16.shape[0] * B16.shape[0]
    cells = a.shape[0] * b.shape[0]
    t_full = dt * full_cells / cells
    return pairs_of(None, A16) / t_full, dt, a.shape[0], b.shape[0]


def omp_threads():
    v = os.environ.get("OMP_NUM_THREADS")
    return int(v) if v else (os.cpu_count() or 1)


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.proc = None
        self.out = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(gpu_index), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            txt, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            txt = ""
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in txt.strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# the dominant kernel's own sources: its counters stand until one of these changes
GEMM_SOURCES = ("gemm_kernel.cu", "ptx.cuh", "common.cuh")


def kernel_digest(files=GEMM_SOURCES):
    h = hashlib.sha1()
    d = os.path.join(ROOT, "contrastive_embedding_loss_gb300", "csrc")
    for f in files:
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload):
    """Per-launch DRAM bytes of the dominant kernel from a committed ncu summary, if it was
    taken on the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(workload)
    except Exception:
        return None
    if not rec or rec.get("kernel_digest") != kernel_digest():
        return None
    return rec.get("dram_bytes_per_launch")


def dist_setup(n_gpus):
    import torch

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist

        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier_max(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_reference(args, rank, world):
    """The reference arm: the float64 oracle on the host cores, rank 0 only."""
    if rank != 0:
        return
    from contrastive_embedding_loss_gb300 import synth

    kind, A16, B16, scale, bias = synth.workload(args.workload)
    rates = []
    for i in range(args.warmup + args.steps):
        r, dt, na, nb = oracle_rate(kind, A16, B16, scale, bias, REFERENCE_STEP_PAIRS)
        if i >= args.warmup:
            rates.append((r, dt))
    value = float(np.mean([r for r, _ in rates]))
    N = A16.shape[0]
    full_t = pairs_of(None, A16) / value
    line = {
        # ms_per_step: the wall time of one timed step as run (one sub-batch); the full batch's
        # time at the oracle's rate is ms_per_step_full_batch
        "impl": "reference", "metric": METRIC, "value": value, "unit": "pairs/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * float(np.mean([dt for _, dt in rates])),
        "ms_per_step_full_batch": 1000 * full_t, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": run_config(args, kind, A16, B16, scale, bias, world),
        "cpu_baseline": {"value": value, "unit": "pairs/s", "cores": omp_threads(), "kind": "oracle",
                         "sample": f"float64 oracle fwd+bwd on the first {REFERENCE_STEP_PAIRS} pairs per step; "
                                   f"time scaled to the full batch by cells ({N}x{B16.shape[0]})"},
        "e2e": {"value": value, "unit": "pairs/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    import torch

    from contrastive_embedding_loss_gb300 import binding, synth

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    assert binding.uf_contrastive_init(local) == binding.UF_OK

    kind, A16, B16, scale, bias = synth.workload(args.workload)
    Na, D = A16.shape
    Nb = B16.shape[0]
    k = binding.KINDS[kind]
    n = len(LADDER)
    to_t = lambda x: torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)  # noqa: E731
    A_h, B_h = to_t(A16).pin_memory(), to_t(B16).pin_memory()
    A_d, B_d = A_h.to(dev), B_h.to(dev)
    ws_bytes = binding.uf_contrastive_workspace_size(Na, Nb, D, LADDER, k, True)
    if args.min_workspace or args.weights_gib is not None:
        extra = int((args.weights_gib or 0.0) * (1 << 30)) // 256 * 256
        ws_bytes = min(ws_bytes, binding.uf_contrastive_workspace_min(Na, Nb, D, LADDER, k, True) + extra)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=dev)
    loss = torch.empty(n, dtype=torch.float32, device=dev)
    dA = torch.empty((Na, D), dtype=torch.float32, device=dev)
    dB = torch.empty((Nb, D), dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    loss_h = torch.empty(n, dtype=torch.float32).pin_memory()
    stream = torch.cuda.current_stream(dev)

    def step(a_ptr, b_ptr):
        st = binding.uf_contrastive_fwd_bwd(a_ptr, b_ptr, Na, Nb, D, LADDER, k, scale, bias, None, loss.data_ptr(),
                                            None, None, dA.data_ptr(), dB.data_ptr(), ws.data_ptr(), ws_bytes,
                                            status.data_ptr(), stream.cuda_stream)
        if st != binding.UF_OK:
            raise binding.UfError(st, "uf_contrastive_fwd_bwd")

    # ---- device-resident timing (inputs 2 x Na*D*2 bytes, larger than the 129 MB L2 at N=65536)
    for _ in range(args.warmup):
        step(A_d.data_ptr(), B_d.data_ptr())
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0])
                          if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    ev0.record(stream)
    for _ in range(args.steps):
        step(A_d.data_ptr(), B_d.data_ptr())
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_local = ev0.elapsed_time(ev1)
    # the same K steps again with the library's per-kernel CUDA events on (two event records
    # around each kernel group, on the call's stream): the kernel split and the dominant
    # kernel's live launch time; kept out of the timed steps above, whose time they would add to
    binding.uf_contrastive_profile(True)
    torch.cuda.synchronize()
    for _ in range(args.steps):
        step(A_d.data_ptr(), B_d.data_ptr())
    torch.cuda.synchronize()
    clk = clocks.stop()
    prof = {binding.KERNEL_GROUPS[g]: binding.uf_contrastive_profile_read(g) for g in range(len(binding.KERNEL_GROUPS))}
    binding.uf_contrastive_profile(False)
    assert int(status.item()) == 0, "a kernel reported a timeout"
    ms = barrier_max(ms_local, world)
    ms_step = ms / args.steps
    units = pairs_of(None, A16)
    value = units * world * args.steps / (ms / 1e3)

    # ---- the same step captured once in a CUDA graph and replayed (the call only enqueues work
    # on the caller's stream, so a training loop can capture it): what launch latency costs
    graph = None
    try:
        g = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                gs = torch.cuda.current_stream(dev)
                st = binding.uf_contrastive_fwd_bwd(A_d.data_ptr(), B_d.data_ptr(), Na, Nb, D, LADDER, k, scale, bias,
                                                    None, loss.data_ptr(), None, None, dA.data_ptr(), dB.data_ptr(),
                                                    ws.data_ptr(), ws_bytes, status.data_ptr(), gs.cuda_stream)
                if st != binding.UF_OK:
                    raise binding.UfError(st, "uf_contrastive_fwd_bwd (captured)")
        stream.wait_stream(side)
        for _ in range(args.warmup):
            g.replay()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        ms_graph = barrier_max(ev0.elapsed_time(ev1), world)
        graph = {"value": units * world * args.steps / (ms_graph / 1e3), "unit": "pairs/s",
                 "ms_per_step": ms_graph / args.steps,
                 "how": "one uf_contrastive_fwd_bwd captured in a CUDA graph, replayed every step"}
        del g
    except Exception as exc:  # capture is reported, not required
        graph = {"error": str(exc)[:200]}
    assert int(status.item()) == 0, "a kernel reported a timeout"

    # ---- end to end through the public API with host buffers: H2D inputs, D2H loss, every step.
    # A training loop's loader copies the next batch while the current one computes, so the
    # inputs are double-buffered on the device: step i + 1's copy (split over COPY_SPLIT
    # streams, so that several copy engines share it) runs during step i, once step i - 1 has
    # released that buffer.  Every step's copy, the first included, lies inside the timed region.
    copy_streams = [torch.cuda.Stream(dev) for _ in range(COPY_SPLIT)]
    bufs = [(A_d, B_d), (torch.empty_like(A_d), torch.empty_like(B_d))]
    free = [torch.cuda.Event(), torch.cuda.Event()]       # the step that last read buffer b is done
    ready = [[torch.cuda.Event() for _ in range(COPY_SPLIT)] for _ in range(2)]  # buffer b's copies are done

    def copy_inputs(bi):
        pieces = []
        for src, dst in ((A_h, bufs[bi][0]), (B_h, bufs[bi][1])):
            per = (src.shape[0] + COPY_SPLIT // 2 - 1) // (COPY_SPLIT // 2)
            pieces += [(src[r0:r0 + per], dst[r0:r0 + per]) for r0 in range(0, src.shape[0], per)]
        for cs in copy_streams:
            cs.wait_event(free[bi])
        for i, (src, dst) in enumerate(pieces):
            with torch.cuda.stream(copy_streams[i % COPY_SPLIT]):
                dst.copy_(src, non_blocking=True)
        for cs, ev in zip(copy_streams, ready[bi]):
            ev.record(cs)

    def e2e_steps(count):
        for bi in range(2):
            free[bi].record(stream)
        copy_inputs(0)
        for i in range(count):
            bi = i % 2
            if i + 1 < count:
                copy_inputs(1 - bi)  # runs during this step
            for ev in ready[bi]:
                stream.wait_event(ev)
            step(bufs[bi][0].data_ptr(), bufs[bi][1].data_ptr())
            free[bi].record(stream)
            loss_h.copy_(loss, non_blocking=True)

    e2e_steps(2)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ev0.record(stream)
    e2e_steps(args.steps)
    ev1.record(stream)
    torch.cuda.synchronize()
    ms_e2e = barrier_max(ev0.elapsed_time(ev1), world)
    e2e_value = units * world * args.steps / (ms_e2e / 1e3)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    peak_tf = float(peaks.get("bf16_tflops_sustained", peaks.get("bf16_tflops")))
    # dominant kernel by device time; its algorithmic flops over its own device time
    dom = max(prof, key=lambda g: prof[g][0])
    dom_ms, dom_pairs, dom_launches = prof[dom]
    per_launch_ms = dom_ms / max(dom_launches, 1)
    alg_step = group_flops(dom, kind, Na, Nb, D, LADDER)
    roof = None
    if alg_step is not None:
        per_launch = args.steps / max(dom_launches, 1)
        alg_launch = alg_step * per_launch
        # the merged path runs a second kernel in the norm-backward group (its row-scalar sums)
        merged = prof["norm_bwd"][2] >= 2 * args.steps
        exe_launch = group_flops_executed(dom, kind, Na, Nb, D, LADDER, merged) * per_launch
        achieved = alg_launch / (per_launch_ms / 1e3) / 1e12
        traffic = ncu_traffic(args.workload)
        alg_bytes = group_bytes(dom, kind, Na, Nb, D, LADDER)
        roof = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": peak_tf, "unit": "TFLOP/s",
                "frac": achieved / peak_tf, "traffic": traffic,
                "peak_source": f"{peak_src} bf16_tflops_sustained",
                "algorithmic_flops_per_launch": alg_launch,
                "executed_flops_per_launch": exe_launch,
                "executed_tflops": exe_launch / (per_launch_ms / 1e3) / 1e12,
                "algorithmic_bytes_per_launch": None if alg_bytes is None else alg_bytes * per_launch,
                "traffic_over_algorithmic": (None if traffic is None or alg_bytes is None
                                             else traffic / (alg_bytes * per_launch)),
                "launches_per_step": dom_launches / args.steps,
                "ms_per_launch": per_launch_ms, "share_of_step": dom_ms / ms_local}
    cflops = credited_flops(kind, Na, Nb, D)
    line = {
        "metric": METRIC, "value": value, "unit": "pairs/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": run_config(args, kind, A16, B16, scale, bias, world),
        "workspace_bytes": int(ws_bytes),
        "tflops_credited": cflops / (ms_step / 1e3) / 1e12,
        "tflops_executed": executed_flops(kind, Na, Nb, D, LADDER, prof["norm_bwd"][2] >= 2 * args.steps)
        / (ms_step / 1e3) / 1e12,
        "frac_credited_of_bf16_peak": cflops / (ms_step / 1e3) / 1e12 / peak_tf,
        "roofline": roof,
        "kernels_ms_per_step": {g: prof[g][0] / args.steps for g in prof},
        "kernels_how": "a second pass of the same steps with per-kernel CUDA events on the call's stream "
                       "(the timed steps run without them)",
        "gpu_launches": int(sum(prof[g][2] for g in prof)),
        "e2e": {"value": e2e_value, "unit": "pairs/s", "h2d_bytes_per_step": int(A_h.numel() * 2 + B_h.numel() * 2),
                "d2h_bytes_per_step": int(loss_h.numel() * 4), "ms_per_step": ms_e2e / args.steps,
                "copies": f"pinned host -> device, split over {COPY_SPLIT} streams, double-buffered: step i + 1's "
                          f"inputs copied during step i (every copy inside the timed region)",
                "results": "the per-prefix loss is copied to pinned host memory every step; dA and dB "
                           f"({2 * (Na + Nb) * D} bytes of fp32) stay on the device, where the training step "
                           "that consumes them runs"},
        "graph": graph,
        "clocks": clk,
    }
    if not args.no_cpu_baseline and world == 1:
        r, dt, na, nb = oracle_rate(kind, A16, B16, scale, bias, ORACLE_SAMPLE_PAIRS)
        line["cpu_baseline"] = {"value": r, "unit": "pairs/s", "cores": omp_threads(), "kind": "oracle",
                                "sample": f"float64 oracle fwd+bwd on the first {na}x{nb} pairs ({dt:.1f} s); "
                                          f"time scaled to {Na}x{Nb} by cells"}
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
