"""GPU parity of the tile-packed NVFP4 operand path, through the C ABI.

* nvfp4_pack_operand against the oracle's byte-by-byte definition of the
  layout (bit for bit, guard bytes past the end untouched);
* nvfp4_gemm_packed against the CPU oracle's NVFP4 GEMM under the GEMM
  tolerance, on shapes whose tails leave the peer CTA's row blocks of A or B
  past M or N (copies skipped there), and on the 16384^3 workload sampled;
* the same GEMM through the tensor-map plan of the same tile shape gives the
  same bits (identical MMA sequence; only the way operands arrive differs).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import block_scaled_precision_persistent_gb300 as bsg
import oracle
import workloads
from test_gemm_gpu import (assert_close, assert_guard, bits, check_sampled_nvfp4, dev, new_out,  # noqa: F401
                           oracle_nvfp4, tile_samples)

pytestmark = pytest.mark.gpu

GUARD = 4096


def pack_gpu(X, rows, K, dev):
    n = bsg.nvfp4_packed_operand_bytes(rows, K)
    assert n == oracle.packed_operand_bytes(rows, K)
    buf = torch.full((n + GUARD,), 0xA5, dtype=torch.uint8, device=dev)
    bsg.nvfp4_pack_operand(rows, K, X, buf[:n])
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    tail = buf[n:].cpu().numpy()
    assert (tail == 0xA5).all(), "pack wrote past the end"
    return buf[:n]


@pytest.mark.parametrize("rows,K", [(1, 256), (127, 512), (128, 256), (300, 768), (513, 1024)])
def test_pack_operand_bit_exact(dev, rows, K):
    g = torch.Generator().manual_seed(rows * 7 + K)
    X = torch.randint(0, 256, (rows, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    got = pack_gpu(X.to(dev), rows, K, dev).cpu().numpy()
    ref = oracle.pack_operand_tiles(X.numpy(), K)
    assert np.array_equal(got, ref)


def swizzled_scales(sf, rows, K, dev):
    out = torch.empty(bsg.nvfp4_swizzled_scale_bytes(rows, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(rows, K, sf, out)
    return out


def gpu_packed(p, dev):
    M, N, K = p["M"], p["N"], p["K"]
    A, B = p["A"].to(dev), p["B"].to(dev)
    Ap, Bp = pack_gpu(A, M, K, dev), pack_gpu(B, N, K, dev)
    sa, sb = swizzled_scales(p["sfA"].to(dev), M, K, dev), swizzled_scales(p["sfB"].to(dev), N, K, dev)
    flat, D = new_out(M, N, dev)
    bsg.nvfp4_gemm_packed(M, N, K, Ap, sa, Bp, sb, p["alpha"], D)
    assert bsg.bsg_last_launch_count() == 1
    assert bsg.bsg_last_plan_name() == "nvfp4_tc2_256x256_s5_acc1_packed"
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert_guard(flat)
    return flat, D, (A, B, sa, sb)


# (M, N): M < 128 and N < 128 leave the peer's A and B row blocks empty;
# 200 x 120 its B block; 300, 392, 520 x 648 ragged tails over several tiles
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1, 8, 256), (200, 120, 512), (300, 392, 768),
                                   (130, 136, 1280), (520, 648, 1024), (777, 1032, 2304)])
def test_gemm_packed_parity(dev, M, N, K):
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
    _, D, _ = gpu_packed(p, dev)
    _, T, ref = oracle_nvfp4(p)
    assert_close(bits(D), ref, T, f"packed {M}x{N}x{K}")


def test_gemm_packed_long_k_alpha(dev):
    """K = 8192 (32 k-blocks per tile, the ring wraps many times), fresh 2^u
    scales on every block, a negative alpha."""
    M, N, K = 384, 512, 8192
    g = torch.Generator().manual_seed(5)
    p = dict(M=M, N=N, K=K, alpha=-0.75,
             A=torch.randint(0, 256, (M, K // 2), generator=g, dtype=torch.int32).to(torch.uint8),
             B=torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.int32).to(torch.uint8),
             sfA=workloads.uniform_nvfp4(M, K, 15, "cpu")[1],
             sfB=workloads.uniform_nvfp4(N, K, 19, "cpu")[1])
    _, D, _ = gpu_packed(p, dev)
    _, T, ref = oracle_nvfp4(p)
    assert_close(bits(D), ref, T, "packed long K")


def test_gemm_packed_matches_tensor_map_plan(dev):
    """Same tile shape, same MMAs: the tensor-map plan gives identical bits."""
    M, N, K = 1000, 776, 1536
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
    _, D, (A, B, sa, sb) = gpu_packed(p, dev)
    flat2, D2 = new_out(M, N, dev)
    bsg.bsg_force_plan("nvfp4_tc2_256x256_s5_acc1")
    try:
        bsg.nvfp4_gemm_swizzled(M, N, K, A, sa, B, sb, p["alpha"], D2)
    finally:
        bsg.bsg_force_plan(None)
    torch.cuda.synchronize()
    assert np.array_equal(bits(D), bits(D2))


def test_packed_plan_not_forceable_elsewhere(dev):
    """The packed plan reads operands only nvfp4_gemm_packed supplies."""
    M = N = K = 256
    A, sfA = workloads.uniform_nvfp4(M, K, 1, dev)
    B, sfB = workloads.uniform_nvfp4(N, K, 2, dev)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    bsg.bsg_force_plan("nvfp4_tc2_256x256_s5_acc1_packed")
    try:
        with pytest.raises(bsg.BsgError) as e:
            bsg.nvfp4_gemm(M, N, K, A, sfA, B, sfB, 1.0, D)
        assert e.value.code == bsg.BSG_ERR_NO_PLAN
    finally:
        bsg.bsg_force_plan(None)


def test_gemm_packed_full_size_sampled(dev):
    """16384^3, the benchmark's workload: sampled rows and columns."""
    w = workloads.WORKLOADS["nvfp4_16384"]
    p = workloads.make_nvfp4(w, dev)
    M, N, K = w.M, w.N, w.K
    flat, D, _ = gpu_packed(p, dev)
    rows, cols = tile_samples(M, N, 128, 256, seed=M + 1)
    rows = rows[::2] + [M - 1]
    check_sampled_nvfp4(p, D, sorted(set(rows)), cols, "packed 16384")
    del flat, D
    torch.cuda.empty_cache()
