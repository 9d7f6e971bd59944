"""Every output of the benchmarked full-size GEMMs, checked against the oracle.

The 16384^3 NVFP4 GEMM and the 8192^3 FP8 GEMM run as the benchmark runs
them (default plan; nvfp4_gemm with row-major scales, fp8_gemm with the
scales folded into alpha). Their results are too large for the element-wise
oracle (hours at 16384^3), so:

  * Freivalds' check covers every element: D x against alpha Adeq (Bdeq^T x)
    for four random +-1 vectors x, with the summed per-element bound and the
    sharper Hoeffding bound (oracle.freivalds_outcome);
  * eight whole 256 x 256 output tiles are compared element by element with
    the oracle: the first and the last, both sides of a rasterisation-group
    boundary (at the first and the last N tile), and both sides of the
    boundary between the persistent kernel's first and second waves.

"Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
Failures", section "The matrix also compared Triton with a reference
implementation": the output is compared with a reference implementation
under a format-specific tolerance.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg
import oracle
import workloads

pytestmark = pytest.mark.gpu

TILE = 256          # the pair plans' output tile
RASTER = 16         # M tiles per rasterisation group (the library's default)


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    bsg.bsg_force_plan(None)
    return d


def raster_coords(tile, m_tiles, n_tiles, group=RASTER):
    """(m tile, n tile) of the tile-th tile in the rasterised order: groups
    of `group` M tiles, M fastest inside a group."""
    per = group * n_tiles
    g, local = divmod(tile, per)
    gm = min(group, m_tiles - g * group)
    return g * group + local % gm, local // gm


def check_tiles(M, N):
    """The eight 256 x 256 tiles named in the module docstring."""
    mt, nt = M // TILE, N // TILE
    waves = torch.cuda.get_device_properties(0).multi_processor_count // 2   # CTA pairs
    tiles = [(0, 0), (mt - 1, nt - 1), (RASTER - 1, 0), (RASTER, 0), (RASTER - 1, nt - 1), (RASTER, nt - 1),
             raster_coords(waves - 1, mt, nt), raster_coords(waves, mt, nt)]
    assert len(set(tiles)) == 8, tiles
    return tiles


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _check(D_bits, rhs, x, tile_ref, what):
    v = oracle.freivalds_outcome(D_bits, x, rhs)
    assert v["finite"], f"{what}: non-finite outputs"
    assert v["ok_summed"], f"{what}: Freivalds summed bound exceeded (worst ratio {v['worst_summed']:.3g})"
    assert v["ok_hoeffding"], (f"{what}: Freivalds Hoeffding bound exceeded (worst ratio "
                               f"{v['worst_hoeffding']:.3g}; first failing (vector, row) {v['fails'][:4]})")
    for (tm, tn), (T, ref) in tile_ref.items():
        got = D_bits[tm * TILE:(tm + 1) * TILE, tn * TILE:(tn + 1) * TILE]
        ok = oracle.within_tolerance(got, ref, T)
        assert ok.all(), f"{what}: tile ({tm},{tn}) has {int((~ok).sum())} outputs outside tolerance"


def test_nvfp4_16384_every_output(dev):
    w = workloads.WORKLOADS["nvfp4_16384"]
    p = workloads.make_nvfp4(w, dev)
    M, N, K = w.M, w.N, w.K
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    bsg.nvfp4_gemm(M, N, K, p["A"], p["sfA"], p["B"], p["sfB"], p["alpha"], D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    Dh = _bits(D)
    del D
    ops = tuple(p[k].cpu().numpy() for k in ("A", "sfA", "B", "sfB"))
    o = oracle.get()
    x = oracle.rademacher(4, N, seed=0xF4E1)
    rhs = o.nvfp4_freivalds(*ops, p["alpha"], K, x)
    tile_ref = {}
    for tm, tn in check_tiles(M, N):
        _, T, ref = o.nvfp4_gemm(*ops, p["alpha"], K, rows=range(tm * TILE, (tm + 1) * TILE),
                                 cols=range(tn * TILE, (tn + 1) * TILE))
        tile_ref[(tm, tn)] = (T, ref)
    _check(Dh, rhs, x, tile_ref, "nvfp4 16384^3")


def test_fp8_8192_every_output(dev):
    w = workloads.WORKLOADS["fp8_8192"]
    q = workloads.make_fp8(w, dev)
    M, N, K = w.M, w.N, w.K
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    bsg.fp8_gemm(M, N, K, q["A"], None, q["B"], None, q["alpha"], D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    Dh = _bits(D)
    A, B = q["A"].cpu().numpy(), q["B"].cpu().numpy()
    o = oracle.get()
    x = oracle.rademacher(4, N, seed=0xF8E1)
    rhs = o.fp8_freivalds(A, B, q["alpha"], x)
    tile_ref = {}
    for tm, tn in check_tiles(M, N):
        _, T, ref = o.fp8_gemm(A, B, q["alpha"], rows=range(tm * TILE, (tm + 1) * TILE),
                               cols=range(tn * TILE, (tn + 1) * TILE))
        tile_ref[(tm, tn)] = (T, ref)
    _check(Dh, rhs, x, tile_ref, "fp8 8192^3")


def test_check_tiles_cover_the_named_boundaries():
    """Host-side: the tile list holds the first and last tiles, both sides of
    the raster-group boundary, and two consecutive tiles of the schedule."""
    mt = nt = 64
    assert raster_coords(0, mt, nt) == (0, 0)
    assert raster_coords(mt * nt - 1, mt, nt) == (mt - 1, nt - 1)
    assert raster_coords(RASTER - 1, mt, nt) == (RASTER - 1, 0)
    assert raster_coords(RASTER, mt, nt) == (0, 1)
    assert raster_coords(RASTER * nt, mt, nt) == (RASTER, 0)
