"""Freivalds' full-product check, on the CPU: it accepts the oracle's own
result (and results perturbed anywhere inside the element-wise tolerance),
and rejects results with a planted mistake -- one flipped BF16 exponent bit,
two swapped 32 x 32 blocks, a dropped K block, a transposed operand, a NaN.

The GPU tests run the same check on every output of the benchmarked
16384^3 NVFP4 and 8192^3 FP8 GEMMs ("Triton #11171 - Why Two New NVFP4 Test
Cases Produced Twelve Tensor-Memory Failures", section "The matrix also
compared Triton with a reference implementation": the output is compared
with a reference under a format-specific tolerance).
"""
from __future__ import annotations

import numpy as np
import pytest

import oracle
import workloads

M, N, K = 384, 512, 1024


@pytest.fixture(scope="module")
def case():
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=M, N=N, K=K)
    ops = tuple(p[k].numpy() for k in ("A", "sfA", "B", "sfB"))
    S, T, D = oracle.get().nvfp4_gemm(*ops, p["alpha"], K)
    x = oracle.rademacher(4, N, seed=0xF5E1)
    rhs = oracle.get().nvfp4_freivalds(*ops, p["alpha"], K, x)
    return dict(ops=ops, alpha=p["alpha"], S=S, T=T, D=D, x=x, rhs=rhs)


def test_accepts_the_oracle_result(case):
    v = oracle.freivalds_outcome(case["D"], case["x"], case["rhs"])
    assert v["ok"], v
    assert v["worst_hoeffding"] < 0.5


def test_accepts_errors_inside_the_tolerance(case):
    """Every nonzero element moved by one BF16 ulp (at most 2^-7 of its
    value, so inside the tolerance), up or down in magnitude at random,
    independently of x: a correct result as far as the contract goes."""
    rng = np.random.default_rng(3)
    D = case["D"].astype(np.int32)
    step = rng.choice([-1, 1], size=D.shape)
    moved = np.where((D & 0x7FFF) != 0, D + step, D).astype(np.uint16)
    assert oracle.within_tolerance(moved, case["D"], case["T"]).all()
    assert (moved != case["D"]).mean() > 0.99
    v = oracle.freivalds_outcome(moved, case["x"], case["rhs"])
    assert v["ok"], v


def test_rejects_one_flipped_exponent_bit(case):
    """One BF16 output bit flipped: bit 10 (exponent bit 3) of one element
    whose bit is clear, so it grows 256-fold."""
    D = case["D"].copy()
    ref = oracle.bf16_bits_to_float(D)
    cand = np.argwhere((np.abs(ref) >= 8.0) & ((D & (1 << 10)) == 0))
    i, j = cand[len(cand) // 2]
    D[i, j] ^= np.uint16(1 << 10)
    v = oracle.freivalds_outcome(D, case["x"], case["rhs"])
    assert not v["ok"] and not v["ok_summed"] and not v["ok_hoeffding"], v
    assert all(row == i for _, row in v["fails"])


def test_rejects_two_swapped_blocks(case):
    """Two 32 x 32 output blocks of one row block exchanged (a tile written
    to the wrong place)."""
    D = case["D"].copy()
    a = D[64:96, 0:32].copy()
    D[64:96, 0:32] = D[64:96, 256:288]
    D[64:96, 256:288] = a
    v = oracle.freivalds_outcome(D, case["x"], case["rhs"])
    assert not v["ok_hoeffding"], v
    assert {row for _, row in v["fails"]} <= set(range(64, 96))


def test_rejects_a_dropped_k_block():
    """The product without its last 16-element block (a planted oracle
    computes it), checked against the real right-hand side."""
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=256, N=256, K=512)
    ops = tuple(p[k].numpy() for k in ("A", "sfA", "B", "sfB"))
    bad = oracle.Oracle(defines=("BSO_MUTANT_DROP_LAST_BLOCK",))
    _, _, D = bad.nvfp4_gemm(*ops, p["alpha"], 512)
    x = oracle.rademacher(4, 256, seed=9)
    v = oracle.freivalds_outcome(D, x, oracle.get().nvfp4_freivalds(*ops, p["alpha"], 512, x))
    assert not v["ok_hoeffding"], v


def test_rejects_a_transposed_operand():
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=256, N=256, K=512)
    ops = tuple(p[k].numpy() for k in ("A", "sfA", "B", "sfB"))
    bad = oracle.Oracle(defines=("BSO_MUTANT_TRANSPOSE_B",))
    _, _, D = bad.nvfp4_gemm(*ops, p["alpha"], 512)
    x = oracle.rademacher(4, 256, seed=10)
    v = oracle.freivalds_outcome(D, x, oracle.get().nvfp4_freivalds(*ops, p["alpha"], 512, x))
    assert not v["ok"], v


def test_rejects_a_nan(case):
    D = case["D"].copy()
    D[5, 7] = 0x7FC1
    v = oracle.freivalds_outcome(D, case["x"], case["rhs"])
    assert not v["ok"] and not v["finite"]


def test_fp8_accepts_and_rejects():
    w = workloads.WORKLOADS["fp8_8192"]
    p = workloads.make_fp8(w, "cpu", M=192, N=256, K=512)
    A, B = p["A"].numpy(), p["B"].numpy()
    _, _, D = oracle.get().fp8_gemm(A, B, p["alpha"])
    x = oracle.rademacher(4, 256, seed=11)
    rhs = oracle.get().fp8_freivalds(A, B, p["alpha"], x)
    assert oracle.freivalds_outcome(D, x, rhs)["ok"]
    D2 = D.copy()
    D2[100:132, 64:96] = D[100:132, 96:128]
    assert not oracle.freivalds_outcome(D2, x, rhs)["ok_hoeffding"]


def test_rejects_vectors_that_are_not_signs(case):
    with pytest.raises(ValueError):
        oracle.freivalds_outcome(case["D"], case["x"] * 2, case["rhs"])
