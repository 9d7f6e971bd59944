"""GPU parity on seeded random shapes, every plan.

Each shape (M from 1 to 700, N a multiple of 8 up to 1120, K a multiple of
the kind's k-block up to 2048 or 3072) is run through the planner's choice
and through every plan forced in turn; a forced plan that cannot take the
shape must refuse it (BSG_ERR_NO_PLAN, nothing launched), and every plan
that runs must agree with the CPU oracle element by element under
|D_gpu - D_ref| <= 2^-7 |D_ref| + 2^-20 T. The two FP8 pair plans, whose
MMAs differ only in how many 256-column halves one of them covers, must
also give the same bits.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_scaled_precision_persistent_gb300 as bsg
import oracle
import workloads
from test_gemm_gpu import (FP8_PLANS, NVFP4_PLANS, SKINNY_PLANS, assert_close, dev,  # noqa: F401
                           gpu_fp8, gpu_nvfp4)

pytestmark = pytest.mark.gpu

WIDE_FP8 = "fp8_tc2_256x512_s4_acc1"


def shapes(kind: str, count: int, seed: int):
    rng = np.random.default_rng(seed)
    kb = 256 if kind == "nvfp4" else 128
    out = []
    for _ in range(count):
        M = int(rng.integers(1, 701))
        N = 8 * int(rng.integers(1, 141))
        K = kb * int(rng.integers(1, (3072 if kind == "nvfp4" else 2048) // kb + 1))
        out.append((M, N, K))
    return out


def run_forced(plan, fn):
    """fn() under a forced plan; None when the plan refuses the shape."""
    bsg.bsg_force_plan(plan)
    try:
        return fn()
    except bsg.BsgError as e:
        assert e.code == bsg.BSG_ERR_NO_PLAN, e
        assert bsg.bsg_last_launch_count() == 0
        return None
    finally:
        bsg.bsg_force_plan(None)


@pytest.mark.parametrize("M,N,K", shapes("nvfp4", 16, 2026))
def test_nvfp4_random_shapes_every_plan(dev, M, N, K):
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
    _, T, ref = oracle.get().nvfp4_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(), p["sfB"].numpy(),
                                        p["alpha"], K)
    ran = {}
    for plan in [None] + NVFP4_PLANS + list(SKINNY_PLANS):
        got = run_forced(plan, lambda: gpu_nvfp4(p, dev, "swizzled"))
        if got is None:
            assert plan is not None and plan in SKINNY_PLANS and M > SKINNY_PLANS[plan], (plan, M)
            continue
        assert_close(got, ref, T, f"nvfp4 {M}x{N}x{K} plan {plan or 'auto'}")
        ran[plan or "auto"] = got
    assert all(q in ran for q in NVFP4_PLANS)


@pytest.mark.parametrize("M,N,K", shapes("fp8", 12, 2027))
def test_fp8_random_shapes_every_plan(dev, M, N, K):
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=M, N=N, K=K)
    _, T, ref = oracle.get().fp8_gemm(q["A"].numpy(), q["B"].numpy(), q["alpha"])
    ran = {}
    for plan in [None] + FP8_PLANS + [WIDE_FP8]:
        got = run_forced(plan, lambda: gpu_fp8(q, dev))
        if got is None:
            assert plan == WIDE_FP8 and N % 256 != 0, (plan, N)
            continue
        assert_close(got, ref, T, f"fp8 {M}x{N}x{K} plan {plan or 'auto'}")
        ran[plan or "auto"] = got
    assert all(q_ in ran for q_ in FP8_PLANS)
    if WIDE_FP8 in ran:
        assert np.array_equal(ran[WIDE_FP8], ran["fp8_tc2_256x256_s6_acc2"]), f"fp8 {M}x{N}x{K}: pair plans disagree"
