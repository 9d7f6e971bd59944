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
