"""GPU parity of the two-level NVFP4 quantiser against the CPU oracle.

Codes, row-major and swizzled block scales, amax and s_g are compared bit for
bit (a quantised code is an integer decided in FP32 on both sides). The
hand-worked case of tests/golden/nvfp4_quantize_case.txt, ragged shapes that
span several 128-row x 256-element tiles, an all-zero matrix, signed zeros,
the full 16384 x 16384 size, an input of more than 2^31 elements, and a
quantise -> GEMM chain are covered.
"""
from __future__ import annotations

from pathlib import Path

import numpy as np
import pytest
import torch

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg
import oracle

pytestmark = pytest.mark.gpu
GOLDEN = Path(__file__).resolve().parent / "golden"


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    return d


def bf16_input(rows, K, seed, std=1.0, device="cpu"):
    g = torch.Generator(device="cpu").manual_seed(seed)
    x = torch.randn((rows, K), generator=g, dtype=torch.float32) * std
    return x.to(torch.bfloat16).to(device)


def gpu_quantize(x: torch.Tensor, dev):
    rows, K = x.shape
    xd = x.to(dev).contiguous()
    packed = torch.full((rows, K // 2), 0xAB, dtype=torch.uint8, device=dev)
    swz = torch.full((bsg.nvfp4_swizzled_scale_bytes(rows, K),), 0xAB, dtype=torch.uint8, device=dev)
    rm = torch.full((rows, K // 16), 0xAB, dtype=torch.uint8, device=dev)
    gl = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
    bsg.nvfp4_quantize(rows, K, xd, packed, swz, rm, gl)
    torch.cuda.synchronize()
    assert bsg.bsg_last_launch_count() == 2
    return packed.cpu().numpy(), rm.cpu().numpy(), swz.cpu().numpy(), gl.cpu().numpy()


def check_against_oracle(x: torch.Tensor, dev):
    rows, K = x.shape
    bits = x.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    o = oracle.get()
    p_ref, sf_ref, amax_ref, sg_ref = o.nvfp4_quantize(bits)
    packed, rm, swz, gl = gpu_quantize(x, dev)
    assert gl[0] == amax_ref and gl[1] == sg_ref, (gl, amax_ref, sg_ref)
    assert np.array_equal(rm, sf_ref), f"row-major scales differ at {np.argwhere(rm != sf_ref)[:4]}"
    assert np.array_equal(packed, p_ref), f"codes differ at {np.argwhere(packed != p_ref)[:4]}"
    assert np.array_equal(swz, o.swizzle_scales(sf_ref, K)), "swizzled scales differ"


def test_quantize_worked_case(dev):
    rows = {}
    for line in (GOLDEN / "nvfp4_quantize_case.txt").read_text().splitlines():
        t = line.split()
        if t and not t[0].startswith("#"):
            rows.setdefault(t[0], []).append(t[1:])
    x = torch.zeros((2, 32), dtype=torch.bfloat16)
    for r in rows["x"]:
        x[int(r[0])] = torch.tensor([float(v) for v in r[1:]], dtype=torch.float32).to(torch.bfloat16)
    packed, rm, _, gl = gpu_quantize(x, dev)
    for r in rows["packed"]:
        assert [int(b, 16) for b in r[1:]] == packed[int(r[0])].tolist(), ("packed", r[0])
    for r in rows["scales"]:
        assert [int(b, 16) for b in r[1:]] == rm[int(r[0])].tolist(), ("scales", r[0])
    assert gl[0] == 6.0 and gl[1] == 448.0
    check_against_oracle(x, dev)


@pytest.mark.parametrize("rows,K", [(1, 16), (3, 48), (37, 1040), (128, 256), (129, 512), (300, 4096),
                                    (1000, 1024), (64, 3072)])
def test_quantize_shapes(dev, rows, K):
    check_against_oracle(bf16_input(rows, K, seed=rows * 31 + K), dev)


def test_quantize_small_std_and_signed_zeros(dev):
    """N(0, 0.02) (the skinny workloads' weights), with -0.0 and +0.0 planted."""
    x = bf16_input(256, 3072, seed=5, std=0.02)
    x[0, :40] = -0.0
    x[1, 7] = 0.0
    x[2, 100:116] = -0.0            # a whole block of -0.0: scale 0, codes 0
    check_against_oracle(x, dev)


def test_quantize_all_zero(dev):
    x = torch.zeros((130, 512), dtype=torch.bfloat16)
    packed, rm, swz, gl = gpu_quantize(x, dev)
    assert gl[0] == 0.0 and gl[1] == 1.0
    assert not packed.any() and not rm.any() and not swz.any()


def test_quantize_full_size(dev):
    """16384 x 16384, every output compared."""
    check_against_oracle(bf16_input(16384, 16384, seed=77), dev)


def test_quantize_then_gemm(dev):
    """BF16 A and B quantised on the GPU and multiplied with alpha =
    1 / (s_gA s_gB): equal to the oracle GEMM over the oracle-quantised
    operands, within the GEMM tolerance."""
    M, N, K = 200, 392, 2048
    a = bf16_input(M, K, seed=1)
    b = bf16_input(N, K, seed=2)
    pa, rma, swa, ga = gpu_quantize(a, dev)
    pb, rmb, swb, gb = gpu_quantize(b, dev)
    alpha = float(np.float32(1.0) / (np.float32(ga[1]) * np.float32(gb[1])))
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    bsg.nvfp4_gemm_swizzled(M, N, K, torch.from_numpy(pa).to(dev), torch.from_numpy(swa).to(dev),
                            torch.from_numpy(pb).to(dev), torch.from_numpy(swb).to(dev), alpha, D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    o = oracle.get()
    qa = o.nvfp4_quantize(a.view(torch.int16).numpy().view(np.uint16))
    qb = o.nvfp4_quantize(b.view(torch.int16).numpy().view(np.uint16))
    _, T, ref = o.nvfp4_gemm(qa[0], qa[1], qb[0], qb[1], alpha, K)
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    assert oracle.within_tolerance(got, ref, T).all()


def test_quantize_beyond_2g_elements(dev):
    """Maximum-size edge: 40960 x 53248 BF16 (2.18e9 elements, 4.4 GB), so
    input and output offsets run past 2^31 elements. N(0,1) data generated on
    the device with the tensor's largest magnitude planted in the last row;
    the oracle quantises sampled rows that include it (so its global scale is
    the whole tensor's) and every output of those rows must match bit for
    bit, in the codes and in both scale layouts."""
    rows, K = 40960, 53248
    g = torch.Generator(device=dev).manual_seed(91)
    x = torch.randn((rows, K), generator=g, device=dev, dtype=torch.float32).to(torch.bfloat16)
    x[rows - 1, K - 7] = -1000.0                 # |x| <= ~7 elsewhere at this size
    packed = torch.empty((rows, K // 2), dtype=torch.uint8, device=dev)
    swz = torch.empty((bsg.nvfp4_swizzled_scale_bytes(rows, K),), dtype=torch.uint8, device=dev)
    rm = torch.empty((rows, K // 16), dtype=torch.uint8, device=dev)
    gl = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
    bsg.nvfp4_quantize(rows, K, x, packed, swz, rm, gl)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    sel = [0, 127, 20479, 40191, 40960 - 129, rows - 1]
    xb = x[sel].contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    o = oracle.get()
    p_ref, sf_ref, amax_ref, sg_ref = o.nvfp4_quantize(xb)
    glh = gl.cpu().numpy()
    assert amax_ref == 1000.0 and glh[0] == amax_ref and glh[1] == sg_ref, (glh, amax_ref, sg_ref)
    assert np.array_equal(packed[sel].cpu().numpy(), p_ref)
    assert np.array_equal(rm[sel].cpu().numpy(), sf_ref)
    # swizzled layout: byte of (row, scale column c) in its 128 x 4 block
    ncb = (K // 16 + 3) // 4
    sw = swz.cpu().numpy()
    for i, r in enumerate(sel):
        c = np.arange(K // 16)
        off = ((r // 128) * ncb + c // 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + c % 4
        assert np.array_equal(sw[off], sf_ref[i]), r
    del x, packed, swz, rm
    torch.cuda.empty_cache()


def gpu_quantize_tiles(x: torch.Tensor, dev):
    rows, K = x.shape
    xd = x.to(dev).contiguous()
    n = bsg.nvfp4_packed_operand_bytes(rows, K)
    tiles = torch.full((n + 256,), 0xAB, dtype=torch.uint8, device=dev)
    swz = torch.full((bsg.nvfp4_swizzled_scale_bytes(rows, K),), 0xAB, dtype=torch.uint8, device=dev)
    gl = torch.full((2,), -1.0, dtype=torch.float32, device=dev)
    bsg.nvfp4_quantize_tiles(rows, K, xd, tiles[:n], swz, None, gl)
    torch.cuda.synchronize()
    assert bsg.bsg_last_launch_count() == 2
    t = tiles.cpu().numpy()
    assert (t[n:] == 0xAB).all(), "quantiser wrote past the tile-packed buffer"
    return t[:n], swz.cpu().numpy(), gl.cpu().numpy()


@pytest.mark.parametrize("rows,K", [(1, 256), (127, 512), (128, 256), (300, 1280), (513, 4096)])
def test_quantize_tiles_against_oracle(dev, rows, K):
    """Codes in the tile-packed layout: the oracle's quantisation followed by
    the oracle's tile packing, bit for bit (padding rows zero); scales and
    the global scale as the row-major entry."""
    x = bf16_input(rows, K, seed=rows + K, std=3.0)
    o = oracle.get()
    p_ref, sf_ref, amax_ref, sg_ref = o.nvfp4_quantize(x.view(torch.int16).numpy().view(np.uint16))
    tiles, swz, gl = gpu_quantize_tiles(x, dev)
    assert gl[0] == amax_ref and gl[1] == sg_ref
    ref = oracle.pack_operand_tiles(p_ref, K)
    assert np.array_equal(tiles, ref), f"tile codes differ at {np.argwhere(tiles != ref)[:4]}"
    assert np.array_equal(swz, o.swizzle_scales(sf_ref, K)), "swizzled scales differ"


def test_quantize_tiles_then_packed_gemm(dev):
    """Activations quantised straight into tiles, weights quantised and
    packed, then nvfp4_gemm_packed: the oracle GEMM over the oracle-quantised
    operands, within the GEMM tolerance."""
    M, N, K = 300, 392, 2048
    a = bf16_input(M, K, seed=11)
    b = bf16_input(N, K, seed=12)
    ta, swa, ga = gpu_quantize_tiles(a, dev)
    pb, rmb, swb, gb = gpu_quantize(b, dev)
    bp = torch.empty(bsg.nvfp4_packed_operand_bytes(N, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_pack_operand(N, K, torch.from_numpy(pb).to(dev), bp)
    alpha = float(np.float32(1.0) / (np.float32(ga[1]) * np.float32(gb[1])))
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    bsg.nvfp4_gemm_packed(M, N, K, torch.from_numpy(ta).to(dev), torch.from_numpy(swa).to(dev), bp,
                          torch.from_numpy(swb).to(dev), alpha, D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    o = oracle.get()
    qa = o.nvfp4_quantize(a.view(torch.int16).numpy().view(np.uint16))
    qb = o.nvfp4_quantize(b.view(torch.int16).numpy().view(np.uint16))
    _, T, ref = o.nvfp4_gemm(qa[0], qa[1], qb[0], qb[1], alpha, K)
    got = D.view(torch.int16).cpu().numpy().view(np.uint16)
    assert oracle.within_tolerance(got, ref, T).all()
