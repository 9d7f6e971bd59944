"""Programmatic dependent launch keeps stream order.

With bsg_set_pdl on, each GEMM lets the next launch on the stream start its
prologue early, and every kernel waits for the previous grid before its first
dependent global access. The test chains two of the library's kernels with a
real data dependency: an NVFP4 GEMM writes D1, then an NVFP4 x dense-BF16
GEMM reads D1 as its BF16 weights. Alpha of the first GEMM flips sign every
iteration, so a second GEMM that read D1 early would see the previous
iteration's values. Its result must equal the same second GEMM run after a
full synchronisation, bit for bit (a check of ordering, not of arithmetic:
parity of both GEMMs is covered elsewhere).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def test_pdl_chain_reads_previous_output(dev):
    M1 = N1 = K1 = 4096                       # D1: [4096][4096] BF16, the second GEMM's B [N2][K2]
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M1, K1), dtype=torch.uint8, device=dev)
    sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N1, K1), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M1, K1, p["sfA"], sa)
    bsg.nvfp4_swizzle_scales(N1, K1, p["sfB"], sb)
    D1 = torch.empty((M1, N1), dtype=torch.bfloat16, device=dev)
    M2, N2, K2 = 512, M1, N1
    q = workloads.make_dense(M2, 8, K2, seed=7, device=dev)     # only A and its scales are used
    sq = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M2, K2), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M2, K2, q["sfA"], sq)
    D2 = torch.empty((M2, N2), dtype=torch.bfloat16, device=dev)
    torch.cuda.synchronize()
    bsg.bsg_set_pdl(True)
    try:
        for it in range(6):
            alpha = p["alpha"] * (1.0 if it % 2 == 0 else -1.0)
            bsg.nvfp4_gemm_swizzled(M1, N1, K1, p["A"], sa, p["B"], sb, alpha, D1)
            bsg.nvfp4_dense_gemm(M2, N2, K2, q["A"], sq, D1, q["alpha"], None, None, None, M2, D2)
        torch.cuda.synchronize()
    finally:
        bsg.bsg_set_pdl(False)
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    got = D2.view(torch.int16).cpu().numpy().copy()
    bsg.nvfp4_dense_gemm(M2, N2, K2, q["A"], sq, D1, q["alpha"], None, None, None, M2, D2)
    torch.cuda.synchronize()
    want = D2.view(torch.int16).cpu().numpy()
    assert np.array_equal(got, want)
    assert np.abs(want).any()


def test_pdl_skinny_and_grouped_chains(dev):
    """Back-to-back skinny split-K and grouped launches under PDL give the
    same bits as without it."""
    w = workloads.WORKLOADS["nvfp4_skinny_m64_n3072_k3072"]
    p = workloads.make_nvfp4(w, dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(w.M, w.K), dtype=torch.uint8, device=dev)
    sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(w.N, w.K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(w.M, w.K, p["sfA"], sa)
    bsg.nvfp4_swizzle_scales(w.N, w.K, p["sfB"], sb)
    outs = []
    for pdl in (False, True):
        bsg.bsg_set_pdl(pdl)
        try:
            Ds = [torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev) for _ in range(8)]
            for D in Ds:
                bsg.nvfp4_gemm_swizzled(w.M, w.N, w.K, p["A"], sa, p["B"], sb, p["alpha"], D)
            torch.cuda.synchronize()
        finally:
            bsg.bsg_set_pdl(False)
        outs.append([D.view(torch.int16).cpu().numpy() for D in Ds])
    for a, b in zip(*outs):
        assert np.array_equal(a, b)


def _quantised(rows, K, seed, dev):
    """NVFP4 codes and swizzled scales of a seeded N(0, 1) BF16 matrix, from
    the library's quantiser (alpha is not needed: the test compares bits)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn((rows, K), generator=g).to(torch.bfloat16).to(dev)
    packed = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    swz = torch.empty(bsg.nvfp4_swizzled_scale_bytes(rows, K), dtype=torch.uint8, device=dev)
    gl = torch.empty(2, dtype=torch.float32, device=dev)
    bsg.nvfp4_quantize(rows, K, x, packed, swz, None, gl)
    return x, packed, swz, gl


@pytest.mark.parametrize("M,N,K,family", [(64, 3072, 12288, "skinny"), (128, 3072, 3072, "tc1"),
                                          (4096, 4096, 1024, "tc2")])
def test_pdl_weights_early_chain(dev, M, N, K, family):
    """bsg_set_pdl(2): the skinny-M and 1-SM kernels read B's codes before
    waiting for the previous kernel (the pair kernel behaves as with 1),
    which here is the quantiser rewriting A's codes and scales every
    iteration (from one of two activation matrices). Each iteration's D must
    equal the GEMM of that iteration's activations run after a full
    synchronisation, bit for bit."""
    xs = [_quantised(M, K, 100 + j, dev)[0] for j in range(2)]
    _, B, sb, _ = _quantised(N, K, 7, dev)
    A = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    gl = torch.empty(2, dtype=torch.float32, device=dev)
    Ds = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(6)]
    torch.cuda.synchronize()
    bsg.bsg_set_pdl(2)
    try:
        for it, D in enumerate(Ds):
            bsg.nvfp4_quantize(M, K, xs[it % 2], A, sa, None, gl)
            bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, 0.25, D)
        torch.cuda.synchronize()
        plan = bsg.bsg_last_plan_name()
    finally:
        bsg.bsg_set_pdl(False)
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert family in plan, plan
    want = []
    for j in range(2):
        bsg.nvfp4_quantize(M, K, xs[j], A, sa, None, gl)
        Dw = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, 0.25, Dw)
        torch.cuda.synchronize()
        want.append(Dw.view(torch.int16).cpu().numpy())
    assert not np.array_equal(want[0], want[1])
    for it, D in enumerate(Ds):
        assert np.array_equal(D.view(torch.int16).cpu().numpy(), want[it % 2]), it


def test_pdl_weights_early_fp8_wide(dev):
    """The same promise on the 512-wide FP8 pair plan, A rewritten by a copy
    kernel before every GEMM: the mode changes no result."""
    M, N, K = 512, 1024, 2048
    g = torch.Generator(device="cpu").manual_seed(11)
    srcs = [(torch.randn((M, K), generator=g) * 0.5).to(torch.float8_e4m3fn).to(dev) for _ in range(2)]
    B = (torch.randn((N, K), generator=g) * 0.5).to(torch.float8_e4m3fn).to(dev)
    A = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    Ds = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(6)]
    torch.cuda.synchronize()
    bsg.bsg_set_pdl(2)
    try:
        for it, D in enumerate(Ds):
            A.copy_(srcs[it % 2])
            bsg.fp8_gemm(M, N, K, A, None, B, None, 1.0, D)
        torch.cuda.synchronize()
        plan = bsg.bsg_last_plan_name()
    finally:
        bsg.bsg_set_pdl(False)
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert plan == "fp8_tc2_256x512_s4_acc1", plan
    want = []
    for j in range(2):
        Dw = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        bsg.fp8_gemm(M, N, K, srcs[j], None, B, None, 1.0, Dw)
        torch.cuda.synchronize()
        want.append(Dw.view(torch.int16).cpu().numpy())
    for it, D in enumerate(Ds):
        assert np.array_equal(D.view(torch.int16).cpu().numpy(), want[it % 2]), it


def test_pdl_weights_early_epilogue_chain(dev):
    """Mode 2 on the skinny kernel's epilogue-variant instantiation: the
    previous kernel rewrites A and this iteration's gamma (a copy kernel),
    the GEMM reads B's codes early and everything else after the wait;
    bias, gamma and a row permutation fused. Every D must equal the
    synchronised GEMM of its iteration, bit for bit."""
    M, N, K = 64, 3072, 12288
    xs = [_quantised(M, K, 300 + j, dev)[0] for j in range(2)]
    _, B, sb, _ = _quantised(N, K, 17, dev)
    g = torch.Generator(device="cpu").manual_seed(5)
    bias = torch.randn(N, generator=g).to(dev)
    gammas = [(torch.rand(M, generator=g) + 0.5).to(dev) for _ in range(2)]
    scatter = torch.randperm(M, generator=g).to(torch.int32).to(dev)
    A = torch.empty((M, K // 2), dtype=torch.uint8, device=dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    gl = torch.empty(2, dtype=torch.float32, device=dev)
    gamma = torch.empty(M, dtype=torch.float32, device=dev)
    Ds = [torch.empty((M, N), dtype=torch.bfloat16, device=dev) for _ in range(6)]
    torch.cuda.synchronize()
    bsg.bsg_set_pdl(2)
    try:
        for it, D in enumerate(Ds):
            bsg.nvfp4_quantize(M, K, xs[it % 2], A, sa, None, gl)
            gamma.copy_(gammas[it % 2])
            bsg.nvfp4_gemm_ex(M, N, K, A, sa, B, sb, 0.25, bias, gamma, scatter, M, D)
        torch.cuda.synchronize()
        plan = bsg.bsg_last_plan_name()
    finally:
        bsg.bsg_set_pdl(False)
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert "skinny" in plan, plan
    want = []
    for j in range(2):
        bsg.nvfp4_quantize(M, K, xs[j], A, sa, None, gl)
        Dw = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        bsg.nvfp4_gemm_ex(M, N, K, A, sa, B, sb, 0.25, bias, gammas[j], scatter, M, Dw)
        torch.cuda.synchronize()
        want.append(Dw.view(torch.int16).cpu().numpy())
    assert not np.array_equal(want[0], want[1])
    for it, D in enumerate(Ds):
        assert np.array_equal(D.view(torch.int16).cpu().numpy(), want[it % 2]), it
