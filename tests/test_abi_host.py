"""Host-side tests of the C ABI (no GPU needed): exports, workspace sizing, argument checks."""
import ctypes
import os
import re

import numpy as np
import pytest

from contrastive_embedding_loss_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
LADDER = (64, 128, 256, 512, 1024)


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_functions():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            txt = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"UF_API\s+[\w\s\*]+?\b(uf_\w+)\s*\(", txt))
    return names


def test_library_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert {"uf_contrastive_fwd_bwd", "uf_contrastive_workspace_size", "uf_contrastive_init",
            "uf_status_name", "uf_contrastive_version"} <= names
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_status_names(lib):
    assert binding.uf_status_name(0) == "ok"
    assert binding.uf_status_name(1) == "invalid-argument"
    assert binding.uf_status_name(5) == "device-timeout"
    assert binding.uf_status_name(99) == "unknown"
    assert binding.uf_contrastive_version() == 100


def test_workspace_size(lib):
    ws = binding.uf_contrastive_workspace_size
    assert ws(256, 256, 1024, LADDER, 0, 1) > 0
    assert ws(256, 256, 1024, LADDER, 0, 1) >= ws(256, 256, 1024, LADDER, 0, 0)
    # invalid requests size to 0
    assert ws(256, 255, 1024, LADDER, 0, 1) == 0      # CLIP needs Na == Nb
    assert ws(256, 100, 1024, LADDER, 2, 1) == 0      # ROWS needs Nb >= Na
    assert ws(256, 100, 1024, LADDER, 1, 1) == 0      # so does SigLIP
    assert ws(256, 700, 1024, LADDER, 1, 1) > 0       # SigLIP with extra negative columns
    assert ws(256, 256, 1000, LADDER, 0, 1) == 0      # D not a multiple of 64
    assert ws(256, 256, 1024, (64, 100), 0, 1) == 0   # prefix not a multiple of 64
    assert ws(256, 256, 1024, (128, 64), 0, 1) == 0   # not increasing
    assert ws(256, 256, 512, LADDER, 0, 1) == 0       # last prefix > D
    assert ws(256, 256, 1024, tuple(range(64, 64 * 10, 64)), 0, 1) == 0  # > 8 prefixes
    assert ws(0, 0, 1024, LADDER, 0, 1) == 0
    assert ws(256, 256, 1024, LADDER, 7, 1) == 0      # unknown kind
    # pure function of the arguments, and it grows with the batch
    assert ws(4096, 4096, 1024, LADDER, 0, 1) == ws(4096, 4096, 1024, LADDER, 0, 1)
    assert ws(65536, 65536, 1024, LADDER, 0, 1) > ws(4096, 4096, 1024, LADDER, 0, 1)
    # the forward alone needs little scratch
    assert ws(65536, 65536, 1024, LADDER, 0, 0) < 2 << 30
    # the backward keeps the bf16 weights of every prefix: at N=65536 all rows fit in one
    # chunk (5 x 65536^2 x 2 bytes = 40 GiB) within the default 48 GiB weight budget
    full = 5 * 65536 * 65536 * 2
    assert full <= ws(65536, 65536, 1024, LADDER, 0, 1) - ws(65536, 65536, 1024, LADDER, 0, 0) < full + (2 << 30)
    # the minimum holds the smallest chunk of weights (128 x 256) and never exceeds the recommendation
    wmin = binding.uf_contrastive_workspace_min
    for N in (1, 300, 4096, 65536):
        assert 0 < wmin(N, N, 1024, LADDER, 0, 1) <= ws(N, N, 1024, LADDER, 0, 1)
    assert wmin(65536, 65536, 1024, LADDER, 0, 1) < (3 << 29)  # vs 40 GiB of weights for one chunk
    assert wmin(256, 255, 1024, LADDER, 0, 1) == 0
    assert wmin(4096, 4096, 1024, LADDER, 0, 0) == ws(4096, 4096, 1024, LADDER, 0, 0)  # no weights forward-only
    # larger batches are cut into chunks: the weight array stays within its budget
    big = 262144
    assert ws(big, big, 1024, LADDER, 0, 1) - ws(big, big, 1024, LADDER, 0, 0) < (48 << 30) + (1 << 30)
    # the smallest chunk of weights is 128 rows of A by 256 rows of B: what the backward adds to
    # the minimum is that chunk and its O(N D) arrays (the transposed operands, 2 x D x N x 2
    # bytes = 256 MiB here), not a full row of weights (5 x 128 x N x 2 bytes per chunk row)
    per_weight_chunk = 5 * 128 * 256 * 2
    extra = wmin(65536, 65536, 1024, LADDER, 0, 1) - wmin(65536, 65536, 1024, LADDER, 0, 0)
    assert 2 * 1024 * 65536 * 2 + per_weight_chunk <= extra < 2 * 1024 * 65536 * 2 + per_weight_chunk + (32 << 20)


def test_workspace_holds_the_merged_prefixes_sums(lib):
    """The recommended workspace adds, for CLIP and ROWS with long contractions and a second
    widest prefix that is a multiple of 512, the partial sums that let the two widest prefixes
    share one weight array: 4 (Na/128) Nb + (4 s + 1) Na + Nb floats (s: the weight pass's column
    split, 2 at N = 65536), as the header states."""
    ws = binding.uf_contrastive_workspace_size
    N = 65536
    plain = (64, 128, 256, 384, 1024)  # second widest not a multiple of 512: nothing merged
    sums = 4 * (4 * (N // 128) * N + (4 * 2 + 1) * N + N)
    assert sums == 539492352  # 0.54 GB
    assert ws(N, N, 1024, LADDER, 0, 1) - ws(N, N, 1024, plain, 0, 1) == sums
    # ROWS (8192 queries, 262144 keys) holds them too; its column sums dominate
    q, k = 8192, 262144
    extra = ws(q, k, 1024, LADDER, 2, 1) - ws(q, k, 1024, plain, 2, 1)
    assert 4 * 4 * (q // 128) * k + 4 * (q + k) <= extra < 4 * 4 * (q // 128) * k + 4 * (q + k) + 4 * 4 * 64 * q
    # SigLIP never merges, nor does a forward-only call (no weights)
    assert ws(N, N, 1024, LADDER, 1, 1) == ws(N, N, 1024, plain, 1, 1)
    assert ws(N, N, 1024, LADDER, 0, 0) == ws(N, N, 1024, plain, 0, 0)


# Fake device addresses for calls that return before any CUDA call: 256-byte aligned, one
# 4 GiB slot per argument so that no two buffers overlap (the library refuses overlapping
# written buffers); the workspace sits above every slot, so its 1 TiB reaches none of them.
F = {name: (i + 1) * (4 << 30) for i, name in enumerate(
    ["A", "B", "loss", "row_terms", "col_terms", "dA", "dB", "d_scale", "d_bias", "scale_dev", "bias_dev",
     "pos_offsets", "pos_ids", "status", "X"])}
WS = 1 << 44
FAKE = F["status"]  # any single aligned address


def _call(**kw):
    args = dict(A=F["A"], B=F["B"], Na=256, Nb=256, D=1024, prefixes=LADDER, kind=0, logit_scale=1 / 0.07,
                bias=0.0, prefix_weights=None, loss_per_prefix=F["loss"], row_terms=None, col_terms=None,
                dA=F["dA"], dB=F["dB"], workspace=WS, workspace_bytes=1 << 40, device_status=None, stream=None)
    args.update(kw)
    return binding.uf_contrastive_fwd_bwd(**args)


def test_workspace_below_the_minimum_is_rejected_on_the_host(lib):
    SMALL = 3
    need = binding.uf_contrastive_workspace_min(256, 256, 1024, LADDER, 0, 1)
    assert _call(workspace_bytes=need - 256) == SMALL
    assert _call(workspace_bytes=0) == SMALL


def test_argument_errors_are_found_on_the_host(lib):
    INV, UNS, SMALL = 1, 2, 3
    assert _call(A=None) == INV
    assert _call(loss_per_prefix=None) == INV
    assert _call(workspace=None) == INV
    assert _call(dB=None) == INV                      # dA and dB go together
    assert _call(A=F["A"] + 2) == INV                 # misaligned
    assert _call(workspace=WS + 16) == INV            # workspace must be 256-byte aligned
    assert _call(dA=F["dA"] + 4) == INV
    assert _call(Nb=255) == INV
    assert _call(prefixes=(64, 64)) == INV
    assert _call(kind=3) == INV
    assert _call(logit_scale=-1.0) == INV
    assert _call(logit_scale=float("nan")) == INV
    assert _call(prefix_weights=[1, 1, float("inf"), 1, 1]) == INV
    assert _call(logit_scale=300.0) == UNS            # beyond the largest supported scale (256)
    assert _call(kind=1, logit_scale=70.0, bias=-20.0) == UNS
    assert _call(workspace_bytes=1024) == SMALL


def test_valid_call_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call() == 4  # UF_CUDA_ERROR, raised by the first CUDA runtime call
    assert binding.uf_contrastive_init(0) == 4


def test_missing_library_fails_loudly(tmp_path):
    with pytest.raises(ImportError):
        binding.load(str(tmp_path / "nope.so"))


def _call_ex(d_logit_scale=F["d_scale"], d_bias=F["d_bias"], **kw):
    args = dict(A=F["A"], B=F["B"], Na=256, Nb=256, D=1024, prefixes=LADDER, kind=0, logit_scale=1 / 0.07,
                bias=0.0, logit_scale_dev=None, bias_dev=None, pos_offsets=None, pos_ids=None, prefix_weights=None,
                loss_per_prefix=F["loss"], row_terms=None, col_terms=None, dA=F["dA"], dB=F["dB"],
                d_logit_scale=d_logit_scale, d_bias=d_bias, workspace=WS, workspace_bytes=1 << 40,
                device_status=None, stream=None)
    args.update(kw)
    return binding.uf_contrastive_fwd_bwd_ex(**args)


def test_scale_gradient_argument_errors_are_found_on_the_host(lib):
    INV, UNS = 1, 2
    assert _call_ex(dA=None, dB=None) == INV                    # they come out of the backward
    assert _call_ex(d_bias=None, dA=None, dB=None) == INV
    assert _call_ex(d_logit_scale=F["d_scale"] + 2) == INV              # fp32 scalars: 4-byte aligned
    assert _call_ex(d_bias=F["d_bias"] + 1) == INV
    assert _call_ex(kind=1, logit_scale=0.0, bias=0.0) == UNS   # SigLIP t = 0: dL/dt is not (sum W cos) / t
    assert _call_ex(kind=1, logit_scale=0.0, bias=0.0, d_logit_scale=None) != UNS  # the bias alone is fine
    # the same checks as the plain entry point still apply
    assert _call_ex(Nb=255) == INV
    assert _call_ex(logit_scale=300.0) == UNS
    # the workspace needed is the same with or without the scalar gradients
    need = binding.uf_contrastive_workspace_min(256, 256, 1024, LADDER, 1, 1)
    assert _call_ex(kind=1, logit_scale=10.0, bias=-10.0, workspace_bytes=need - 256) == 3


def test_valid_scale_gradient_call_without_gpu_reports_cuda_error(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call_ex() == 4
    assert _call_ex(kind=1, logit_scale=10.0, bias=-10.0) == 4


def test_device_scalars_are_checked_on_the_host_only_for_alignment(lib):
    INV, CUDA = 1, 4
    assert _call_ex(logit_scale_dev=F["scale_dev"] + 2) == INV
    assert _call_ex(bias_dev=F["bias_dev"] + 1) == INV
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # a host value that would be refused is ignored when the device holds the scalar: the
    # call gets as far as the first CUDA call
    assert _call_ex(logit_scale=float("nan"), logit_scale_dev=F["scale_dev"]) == CUDA
    assert _call_ex(logit_scale=1000.0, logit_scale_dev=F["scale_dev"]) == CUDA
    assert _call_ex(kind=1, logit_scale=70.0, bias=-20.0, bias_dev=F["bias_dev"]) == CUDA
    # large host scales take the max-shifted path instead of being refused
    assert _call_ex(logit_scale=100.0) == CUDA
    assert _call_ex(logit_scale=256.0) == CUDA


def test_label_arguments_are_checked_on_the_host(lib):
    INV, UNS, CUDA = 1, 2, 4
    sig = dict(kind=1, logit_scale=10.0, bias=-10.0)
    assert _call_ex(pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"]) == UNS          # CLIP: no labelled positives
    assert _call_ex(kind=2, logit_scale=20.0, pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"]) == UNS
    assert _call_ex(pos_offsets=F["pos_offsets"], **sig) == INV                  # offsets and ids go together
    assert _call_ex(pos_ids=F["pos_ids"], **sig) == INV
    assert _call_ex(pos_offsets=F["pos_offsets"] + 4, pos_ids=F["pos_ids"], **sig) == INV  # int64 offsets: 8-byte aligned
    assert _call_ex(pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"] + 2, **sig) == INV
    assert _call_ex(Nb=200, **sig) == INV                            # SigLIP needs Nb >= Na
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert _call_ex(pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"], **sig) == CUDA
    assert _call_ex(Nb=700, **sig) == CUDA                           # extra negative columns


def test_oneset_arguments_are_checked_on_the_host(lib):
    INV, UNS, CUDA = 1, 2, 4
    args = dict(X=F["X"], N=256, D=1024, prefixes=LADDER, logit_scale=10.0, bias=-10.0, logit_scale_dev=None,
                bias_dev=None, pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"], prefix_weights=None,
                loss_per_prefix=F["loss"], row_terms=None, dX=F["dA"], d_logit_scale=None, d_bias=None, workspace=WS,
                workspace_bytes=1 << 40, device_status=None, stream=None)
    call = lambda **kw: binding.uf_contrastive_oneset_fwd_bwd(**{**args, **kw})  # noqa: E731
    assert call(pos_offsets=None) == INV           # a one-set batch names its pairs
    assert call(pos_ids=None) == INV
    assert call(X=None) == INV
    assert call(X=F["X"] + 2) == INV
    assert call(logit_scale=70.0, bias=-20.0) == UNS
    assert call(d_logit_scale=F["d_scale"], dX=None) == INV  # the scalar gradients come out of the backward
    need = binding.uf_contrastive_workspace_min(256, 256, 1024, LADDER, 1, 1)
    assert call(workspace_bytes=need - 256) == 3
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert call() == CUDA
    assert call(dX=None) == CUDA


def test_wait_selftest_arguments(lib):
    INV, CUDA = 1, 4
    assert binding.uf_contrastive_selftest_wait(None, 100, None) == INV
    assert binding.uf_contrastive_selftest_wait(FAKE + 2, 100, None) == INV
    assert binding.uf_contrastive_selftest_wait(FAKE, 0, None) == INV
    assert binding.uf_contrastive_selftest_wait(FAKE, 10001, None) == INV
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    assert binding.uf_contrastive_selftest_wait(FAKE, 100, None) == CUDA


C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "uf_contrastive.h"

int main(void) {
  const int ladder[5] = {64, 128, 256, 512, 1024};
  size_t ws = uf_contrastive_workspace_size(256, 256, 1024, ladder, 5, UF_LOSS_CLIP_SYMMETRIC, 1);
  size_t wmin = uf_contrastive_workspace_min(256, 256, 1024, ladder, 5, UF_LOSS_CLIP_SYMMETRIC, 1);
  size_t bad = uf_contrastive_workspace_size(256, 255, 1024, ladder, 5, UF_LOSS_CLIP_SYMMETRIC, 1);
  float loss[5];
  uf_status_t st = uf_contrastive_fwd_bwd(NULL, NULL, 256, 256, 1024, ladder, 5, UF_LOSS_CLIP_SYMMETRIC,
                                          14.0f, 0.0f, NULL, loss, NULL, NULL, NULL, NULL, NULL, 0, NULL, NULL);
  printf("%d %s %zu %zu %zu %d %s\n", uf_contrastive_version(), uf_status_name(UF_DEVICE_TIMEOUT), ws, wmin, bad,
         (int)st, uf_status_name(st));
  return 0;
}
"""


def test_header_compiles_and_links_as_plain_c(lib, tmp_path):
    """The boundary is plain C99: the header compiles with gcc -std=c99 -Wall -Werror, a C
    program links against the library and calls the entry points that need no GPU."""
    import shutil
    import subprocess

    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    so = binding.library_path()
    src = tmp_path / "abi.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi"
    subprocess.check_call(["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I",
                           os.path.join(root, "include"), str(src), "-o", str(exe), so,
                           "-Wl,-rpath," + os.path.dirname(so)])
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    version, timeout_name, ws, wmin, bad, st, st_name = out.stdout.split()
    assert int(version) == binding.uf_contrastive_version()
    assert timeout_name == "device-timeout"
    assert int(ws) == binding.uf_contrastive_workspace_size(256, 256, 1024, (64, 128, 256, 512, 1024), 0, True)
    assert 0 < int(wmin) <= int(ws) and int(bad) == 0  # CLIP needs Na == Nb
    assert int(st) == 1 and st_name == "invalid-argument"  # NULL inputs are refused on the host


def test_overlapping_buffers_are_refused_on_the_host(lib):
    INV, CUDA = 1, 4
    n, Na, D = len(LADDER), 256, 1024
    dA_end = F["dA"] + Na * D * 4
    assert _call(dB=F["dA"] + 256) == INV                          # two outputs share bytes
    assert _call(dA=F["A"]) == INV                                 # an output over an input
    assert _call(dB=F["B"] + 4096) == INV
    assert _call(loss_per_prefix=WS + 1024) == INV                 # an output inside the workspace
    assert _call(device_status=F["dA"] + 64) == INV                # the status word inside an output
    assert _call(workspace=F["dA"], workspace_bytes=1 << 30) == INV
    assert _call(row_terms=F["row_terms"], col_terms=F["row_terms"] + n * Na * 4 - 4) == INV
    assert _call_ex(d_bias=F["d_scale"]) == INV                    # the two scalar gradients
    assert _call_ex(kind=1, logit_scale=10.0, bias=-10.0, pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"],
                    loss_per_prefix=F["pos_offsets"] + 8 * Na) == INV  # the loss over the label offsets' last entry
    assert _call_ex(logit_scale_dev=F["dA"] + 128) == INV          # a device scalar inside an output
    oneset = dict(X=F["X"], N=Na, D=D, prefixes=LADDER, logit_scale=10.0, bias=-10.0, logit_scale_dev=None,
                  bias_dev=None, pos_offsets=F["pos_offsets"], pos_ids=F["pos_ids"], prefix_weights=None,
                  loss_per_prefix=F["loss"], row_terms=None, dX=F["X"], d_logit_scale=None, d_bias=None,
                  workspace=WS, workspace_bytes=1 << 40, device_status=None, stream=None)
    assert binding.uf_contrastive_oneset_fwd_bwd(**oneset) == INV  # dX over the set itself
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    # what is allowed: inputs that overlap (A == B), and buffers that touch without sharing a byte
    assert _call(B=F["A"]) == CUDA
    assert _call(dB=dA_end) == CUDA
    assert _call(loss_per_prefix=WS - n * 4) == CUDA
    assert _call(device_status=dA_end + Na * D * 4) == CUDA  # free memory past the end of dA


def test_binding_checks_shapes_before_anything_else(lib):
    """The binding refuses malformed tensors itself: the C ABI takes D from one matrix and
    would read the other with that row length."""
    import torch

    A = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="same width"):
        binding.contrastive_fwd_bwd(A, torch.zeros(4, 64, dtype=torch.bfloat16))
    with pytest.raises(ValueError, match="2-D"):
        binding.contrastive_fwd_bwd(A[0], A)
    with pytest.raises(ValueError, match="2-D"):
        binding.oneset_fwd_bwd(A[0], (np.zeros(5, np.int64), np.zeros(0, np.int32)))
    with pytest.raises(TypeError, match="CUDA"):
        binding.contrastive_fwd_bwd(A, A)  # host tensors: no CPU path
    with pytest.raises(TypeError, match="CUDA"):
        binding.oneset_fwd_bwd(A, (np.zeros(5, np.int64), np.zeros(0, np.int32)))


def _largest_n_in_static_array(kind, limit):
    lo, hi = 1, 1 << 20
    while lo < hi:
        m = (lo + hi + 1) // 2
        need = binding.uf_contrastive_workspace_min(m, m, 1024, LADDER, kind, 1)
        if need and need <= limit:
            lo = m
        else:
            hi = m - 1
    return lo


def test_static_entry_bounds_match_its_documentation(lib):
    """The header states the largest N that the no-allocation entry point's fixed scratch array
    takes (D = 1024, five prefixes, Na = Nb = N, with gradients); those figures come from
    uf_contrastive_workspace_min, and this pins them."""
    hdr = open(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                            "uf_contrastive.h")).read()
    limit = int(re.search(r"#define UF_STATIC_WORKSPACE_BYTES \((\d+)u << 20\)", hdr).group(1)) << 20
    m = re.search(r"CLIP fits up to N = (\d+),\s*\*\s*SigLIP up to N = (\d+)", hdr)
    assert m, "the header no longer states the bounds"
    assert _largest_n_in_static_array(0, limit) == int(m.group(1))
    assert _largest_n_in_static_array(1, limit) == int(m.group(2))
    # one row more does not fit, and the entry point refuses it on the host
    n = int(m.group(1)) + 1
    assert binding.uf_contrastive_workspace_min(n, n, 1024, LADDER, 0, 1) > limit
