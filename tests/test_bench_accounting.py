"""bench.py's flop and byte accounting, on the CPU.

The roofline fraction the benchmark reports divides the method's own contraction work by the
GEMM time, and the whole-step rates count the tensor work the kernels execute.  These tests pin
those counts to their closed forms for the benchmark workload (N = 65536, D = 1024, prefixes
{64, 128, 256, 512, 1024}) so that a change to the accounting cannot silently move the reported
fractions.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402

N, D = 65536, 1024
PRE = (64, 128, 256, 512, 1024)


def test_method_flops_of_the_gradient_contractions():
    # each of the two contractions contracts every output dimension once: 2 N^2 D
    assert bench.group_flops("gemm", "clip", N, N, D, PRE) == 2 * 2 * N * N * D
    # a score pass sweeps K once for all nested prefixes
    assert bench.group_flops("fwd_tile", "clip", N, N, D, PRE) == 2 * N * N * D
    assert bench.group_flops("bwd_tile", "clip", N, N, D, PRE) == 2 * N * N * D
    assert bench.group_flops("prep", "clip", N, N, D, PRE) is None


def test_executed_flops_prefix_expanded_and_merged():
    # prefix-expanded: prefix k contributes its own p_k dimensions, sum 1984
    assert sum(PRE) == 1984
    assert bench.group_flops_executed("gemm", "clip", N, N, D, PRE) == 2 * 2 * N * N * 1984
    # merged: prefix n-1 runs only above p_{n-2} = 512, so 1984 - 512 = 1472 dimensions
    assert bench.group_flops_executed("gemm", "clip", N, N, D, PRE, merged=True) == 2 * 2 * N * N * 1472
    # the whole step: forward and weight score passes plus both merged contractions = 9984 N^2
    assert bench.executed_flops("clip", N, N, D, PRE, merged=True) == 9984 * N * N
    # SigLIP has no forward score pass (its loss comes out of the weight pass)
    assert bench.executed_flops("siglip", N, N, D, PRE) == 2 * N * N * D + 2 * 2 * N * N * 1984


def test_credited_flops_and_algorithmic_bytes():
    assert bench.credited_flops("clip", N, N, D) == 8 * N * N * D
    assert bench.credited_flops("rows", 8192, 262144, D) == 8 * 8192 * 262144 * D
    assert bench.credited_flops("siglip", N, N, D) == 6 * N * N * D
    # a contraction writes its fp32 gradient once and reads the other side's bf16 rows once;
    # both contractions of a step: 805306368 bytes at the benchmark size (402653184 a launch)
    assert bench.group_bytes("gemm", "clip", N, N, D, PRE) == (4 + 2) * (N + N) * D == 805306368
    assert bench.group_bytes("fwd_tile", "clip", N, N, D, PRE) is None


@pytest.mark.parametrize("pre,dims", [((1024,), 1024), ((512, 1024), 1024), ((64, 256, 1024, 4096), 64 + 256 + 4096)])
def test_merged_count_for_other_ladders(pre, dims):
    # merged: every prefix but the second widest contributes its dimensions (one prefix: no merge)
    assert bench.group_flops_executed("gemm", "clip", 3, 5, pre[-1], pre, merged=True) == 2 * 2 * 3 * 5 * dims


def test_l2_statement_follows_the_input_size():
    import numpy as np

    def rows(n, d=1024):
        return np.zeros((n, d), dtype=np.uint16)

    # the benchmark workload: A and B are 2 x 134 MB, larger than L2
    assert bench.l2_policy(rows(65536), rows(65536)) == "inputs larger than L2 (no flush)"
    # ROWS: 8192 queries and 262144 keys
    assert bench.l2_policy(rows(8192), rows(262144)) == "inputs larger than L2 (no flush)"
    # the small configurations fit in L2, and the line says so
    assert bench.l2_policy(rows(4096), rows(4096)).startswith("inputs (17 MB) fit in L2")
    assert bench.l2_policy(rows(16384), rows(16384)).startswith("inputs (67 MB) fit in L2")
