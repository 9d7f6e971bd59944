"""GPU parity: the CUDA path, called through the C ABI, against the CPU oracle.

Element-by-element comparison under |D_gpu - D_ref| <= 2^-7 |D_ref| + 2^-20 T
(T = sum_k |alpha a sA b sB|); the scale swizzle and the one-hot decode probes
are compared bit for bit. Small and ragged shapes are checked in full; the
full-size workloads (4096^3, 16384^3 NVFP4, 8192^3 FP8), in the launch
configuration the benchmark times, are checked on sampled rows and columns
that touch every output tile.
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

SENTINEL = 0x7FC1          # a NaN pattern no correct output can have
GUARD = 256                # sentinel elements written past the end of D

E2M1 = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6])


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    bsg.bsg_force_plan(None)
    return d


def new_out(M, N, dev):
    """D with a sentinel-filled guard tail; returns (flat buffer, D view)."""
    flat = torch.full((M * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    return flat, flat[: M * N].view(torch.bfloat16).view(M, N)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def assert_guard(flat):
    tail = bits(flat[-GUARD:])
    assert (tail == SENTINEL).all(), "kernel wrote past the end of D"


def assert_close(got, ref, T, what):
    ok = oracle.within_tolerance(got, ref, T)
    if not ok.all():
        bad = np.argwhere(~ok)
        i, j = bad[0]
        g = oracle.bf16_bits_to_float(got[i, j])
        r = oracle.bf16_bits_to_float(ref[i, j])
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} outside tolerance; first at "
                             f"({i},{j}) gpu={g} ref={r} T={T[i, j]}")


def gpu_nvfp4(p, dev, entry="rowmajor", stream=None):
    M, N, K = p["M"], p["N"], p["K"]
    t = {k: p[k].to(dev) for k in ("A", "sfA", "B", "sfB")}
    flat, D = new_out(M, N, dev)
    if entry == "rowmajor":
        bsg.nvfp4_gemm(M, N, K, t["A"], t["sfA"], t["B"], t["sfB"], p["alpha"], D, stream)
        assert bsg.bsg_last_launch_count() == 2      # both scale swizzles in one launch, then the GEMM
    else:
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, t["sfA"], sa, stream)
        bsg.nvfp4_swizzle_scales(N, K, t["sfB"], sb, stream)
        bsg.nvfp4_gemm_swizzled(M, N, K, t["A"], sa, t["B"], sb, p["alpha"], D, stream)
        assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert_guard(flat)
    return bits(D)


def oracle_nvfp4(p, rows=None, cols=None):
    cpu = {k: (p[k].cpu().numpy() if torch.is_tensor(p[k]) else p[k]) for k in ("A", "sfA", "B", "sfB")}
    return oracle.get().nvfp4_gemm(cpu["A"], cpu["sfA"], cpu["B"], cpu["sfB"], p["alpha"], p["K"],
                                   rows=rows, cols=cols)


NVFP4_PLANS = ["nvfp4_tc1_128x256_s3_acc1", "nvfp4_tc1_128x128_s5_acc2",
               "nvfp4_tc2_256x256_s5_acc1", "nvfp4_tc2_256x128_s6_acc2"]
FP8_PLANS = ["fp8_tc1_128x256_s4_acc2", "fp8_tc1_128x128_s6_acc2", "fp8_tc2_256x256_s6_acc2"]


@pytest.fixture(params=[None] + NVFP4_PLANS, ids=["auto"] + NVFP4_PLANS)
def nvfp4_plan(request, dev):
    bsg.bsg_force_plan(request.param)
    yield request.param
    bsg.bsg_force_plan(None)


@pytest.fixture(params=[None] + FP8_PLANS, ids=["auto"] + FP8_PLANS)
def fp8_plan(request, dev):
    bsg.bsg_force_plan(request.param)
    yield request.param
    bsg.bsg_force_plan(None)


# ---------------------------------------------------------------------------
# Scale swizzle: bit-exact
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("rows,K", [(1, 16), (127, 48), (129, 64), (300, 1040), (256, 256),
                                    (300, 512), (4096, 4096), (1000, 16384)])
def test_swizzle_bit_exact(dev, rows, K):
    rng = np.random.default_rng(rows * 7 + K)
    sf = rng.integers(0, 256, (rows, K // 16)).astype(np.uint8)
    want = oracle.get().swizzle_scales(sf, K)
    out = torch.full((want.size,), 0xAB, dtype=torch.uint8, device=dev)   # padding must be zeroed
    bsg.nvfp4_swizzle_scales(rows, K, torch.from_numpy(sf).to(dev), out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want)


@pytest.mark.parametrize("M,N,K", [(1, 300, 16), (127, 129, 48), (300, 8, 1040), (4096, 1000, 4096),
                                   (16384, 16384, 16384)])
def test_swizzle_two_operands_bit_exact(dev, M, N, K):
    """nvfp4_swizzle_scales2: both operands in one launch, each exactly the
    oracle's layout (padding zeroed), guard bytes untouched."""
    rng = np.random.default_rng(M * 3 + N + K)
    sa = rng.integers(0, 256, (M, K // 16)).astype(np.uint8)
    sb = rng.integers(0, 256, (N, K // 16)).astype(np.uint8)
    o = oracle.get()
    wa, wb = o.swizzle_scales(sa, K), o.swizzle_scales(sb, K)
    buf = torch.full((wa.size + wb.size + 512,), 0xAB, dtype=torch.uint8, device=dev)
    oa, ob = buf[: wa.size], buf[wa.size + 256: wa.size + 256 + wb.size]
    bsg.nvfp4_swizzle_scales2(M, N, K, torch.from_numpy(sa).to(dev), oa, torch.from_numpy(sb).to(dev), ob)
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    h = buf.cpu().numpy()
    assert np.array_equal(h[: wa.size], wa)
    assert np.array_equal(h[wa.size + 256: wa.size + 256 + wb.size], wb)
    assert (h[wa.size: wa.size + 256] == 0xAB).all() and (h[wa.size + 256 + wb.size:] == 0xAB).all()


def test_swizzle_two_operands_past_grid_limit(dev):
    """ceil(M/128) + ceil(N/128) = 65536 block rows exceed one launch's grid
    rows: the two operands then take a launch each, with the same result.
    K = 16 keeps it small (8 MiB of scales, 32 MiB swizzled)."""
    M, N, K = 65535 * 128, 128, 16
    rng = np.random.default_rng(5)
    sa = rng.integers(0, 256, (M, 1)).astype(np.uint8)
    sb = rng.integers(0, 256, (N, 1)).astype(np.uint8)
    o = oracle.get()
    wa, wb = o.swizzle_scales(sa, K), o.swizzle_scales(sb, K)
    oa = torch.full((wa.size,), 0xAB, dtype=torch.uint8, device=dev)
    ob = torch.full((wb.size,), 0xAB, dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales2(M, N, K, torch.from_numpy(sa).to(dev), oa, torch.from_numpy(sb).to(dev), ob)
    assert bsg.bsg_last_launch_count() == 2
    torch.cuda.synchronize()
    assert np.array_equal(oa.cpu().numpy(), wa)
    assert np.array_equal(ob.cpu().numpy(), wb)


@pytest.mark.parametrize("offset", [1, 4, 8])
def test_swizzle_unaligned_input(dev, offset):
    """Row-major scales that start off a 16-byte boundary (a sliced buffer):
    the kernel takes its byte path and the result is still bit-exact."""
    rows, K = 300, 4096
    rng = np.random.default_rng(offset)
    sf = rng.integers(0, 256, (rows, K // 16)).astype(np.uint8)
    want = oracle.get().swizzle_scales(sf, K)
    buf = torch.zeros(sf.size + 64, dtype=torch.uint8, device=dev)
    buf[offset:offset + sf.size] = torch.from_numpy(sf.reshape(-1)).to(dev)
    out = torch.full((want.size,), 0xAB, dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(rows, K, buf[offset:], out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), want)


# ---------------------------------------------------------------------------
# NVFP4
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("entry", ["rowmajor", "swizzled"])
def test_nvfp4_uniform_256(dev, nvfp4_plan, entry):
    """The 256^3 workload: all 16 codes, 2^u block scales, full comparison."""
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_256"], "cpu")
    got = gpu_nvfp4(p, dev, entry)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, f"nvfp4 256^3 {entry}")


def test_nvfp4_worked_case(dev, nvfp4_plan):
    """The hand-worked 2x2x32 case (D = [[96, 54], [-48, -27]]) padded with
    zero codes to K = 256 and zero rows to N = 8: exact on the GPU."""
    K, M, N = 256, 2, 8
    codes_a = np.zeros((M, K), np.uint8)
    codes_b = np.zeros((N, K), np.uint8)
    codes_a[0, :32], codes_a[1, :32] = 0x2, 0xA
    codes_b[0, :32] = 0x4
    codes_b[1, :32] = [k % 8 for k in range(32)]
    sfA = np.full((M, K // 16), 0x38, np.uint8)
    sfB = np.full((N, K // 16), 0x38, np.uint8)
    sfA[0, :2], sfA[1, :2] = (0x38, 0x40), (0x30, 0x38)
    sfB[1, :2] = (0x38, 0x28)
    pk = lambda c: torch.from_numpy((c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8))  # noqa: E731
    p = dict(M=M, N=N, K=K, A=pk(codes_a), sfA=torch.from_numpy(sfA), B=pk(codes_b),
             sfB=torch.from_numpy(sfB), alpha=1.0)
    got = oracle.bf16_bits_to_float(gpu_nvfp4(p, dev))
    want = np.zeros((M, N))
    want[:, :2] = [[96, 54], [-48, -27]]
    assert np.array_equal(got, want), got


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (200, 136, 512)])
def test_nvfp4_one_hot_decode(dev, nvfp4_plan, M, N, K):
    """A row i one-hot at k = pi(i) (value 1.0, unit scales): D[i][j] must be
    exactly the E2M1 value of B[j][pi(i)] -- every code, both nibbles."""
    rng = np.random.default_rng(M + N + K)
    pi = np.concatenate([rng.permutation(K) for _ in range(-(-M // K))])[:M]
    codes_a = np.zeros((M, K), np.uint8)
    codes_a[np.arange(M), pi] = 0x2
    codes_b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    pk = lambda c: torch.from_numpy((c[:, 0::2] | (c[:, 1::2] << 4)).astype(np.uint8))  # noqa: E731
    p = dict(M=M, N=N, K=K, A=pk(codes_a), sfA=torch.full((M, K // 16), 0x38, dtype=torch.uint8),
             B=pk(codes_b), sfB=torch.full((N, K // 16), 0x38, dtype=torch.uint8), alpha=1.0)
    got = oracle.bf16_bits_to_float(gpu_nvfp4(p, dev))
    want = E2M1[codes_b[:, pi]].T
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,N,K", [(1, 8, 256), (200, 328, 512), (257, 392, 768), (130, 136, 1280),
                                   (64, 3072, 3072), (520, 648, 1024)])
def test_nvfp4_ragged(dev, nvfp4_plan, M, N, K):
    """Tails in M and N (TMA zero fill and store clipping), several k-blocks."""
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
    got = gpu_nvfp4(p, dev)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, f"nvfp4 {M}x{N}x{K}")


@pytest.mark.parametrize("rep", [0, 1])
def test_nvfp4_long_k(dev, nvfp4_plan, rep):
    """K = 16384 (64 ring stages per tile, every stage with fresh 2^u scales),
    full comparison: exercises the scale-copy / MMA ordering on every stage."""
    w = workloads.WORKLOADS["nvfp4_256"]
    g = torch.Generator().manual_seed(77 + rep)
    M, N, K = 384, 512, 16384
    p = dict(M=M, N=N, K=K, alpha=1.0,
             A=torch.randint(0, 256, (M, K // 2), generator=g, dtype=torch.int32).to(torch.uint8),
             B=torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.int32).to(torch.uint8),
             sfA=workloads.uniform_nvfp4(M, K, 5 + rep, "cpu")[1],
             sfB=workloads.uniform_nvfp4(N, K, 9 + rep, "cpu")[1])
    del w
    got = gpu_nvfp4(p, dev, "swizzled")
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, f"nvfp4 long K rep {rep}")


def test_nvfp4_multi_tile_alpha(dev):
    """512 x 768 x 2048, N(0,1)-quantised, a negative non-unit alpha."""
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=512, N=768, K=2048)
    p["alpha"] = -3.0 * p["alpha"]
    for entry in ("rowmajor", "swizzled"):
        got = gpu_nvfp4(p, dev, entry)
        _, T, ref = oracle_nvfp4(p)
        assert_close(got, ref, T, f"nvfp4 512x768x2048 {entry}")


def tile_samples(M, N, bm, bn, seed):
    """One sampled row per M tile and one sampled column per N tile, at
    varying offsets inside the tile (so every output tile is touched)."""
    rng = np.random.default_rng(seed)
    rows = [min(M - 1, t * bm + int(rng.integers(0, bm))) for t in range(-(-M // bm))]
    cols = [min(N - 1, t * bn + int(rng.integers(0, bn))) for t in range(-(-N // bn))]
    rows = sorted(set(rows) | {0, M - 1})
    cols = sorted(set(cols) | {0, N - 1})
    return rows, cols


def check_sampled_nvfp4(p, D, rows, cols, what):
    Dh = bits(D)
    _, T, ref = oracle_nvfp4(p, rows=rows)
    assert_close(Dh[rows], ref, T, f"{what} sampled rows")
    _, T, ref = oracle_nvfp4(p, cols=cols)
    assert_close(Dh[:, cols], ref, T, f"{what} sampled cols")


def test_nvfp4_output_beyond_2g_elements(dev):
    """Maximum-size edge: D holds more than 2^31 elements (47104^2 BF16,
    4.4 GB), so output offsets run past 4 GB. Default plan through the
    row-major entry; rows across the whole range (first, last, and tile rows
    near the 2^31-element boundary) and columns against the oracle, and the
    guard tail untouched."""
    M = N = 47104
    K = 256
    A, sfA = workloads.uniform_nvfp4(M, K, 71, dev)
    B, sfB = workloads.uniform_nvfp4(N, K, 72, dev)
    p = dict(M=M, N=N, K=K, A=A, sfA=sfA, B=B, sfB=sfB, alpha=0.5)
    flat, D = new_out(M, N, dev)
    bsg.nvfp4_gemm(M, N, K, A, sfA, B, sfB, p["alpha"], D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert_guard(flat)
    boundary = (1 << 31) // N                     # first row whose elements lie past 2^31
    rows = [0, 255, boundary - 1, boundary, boundary + 1, 45311, M - 1]
    cols = [0, 127, 31000, N - 1]
    _, T, ref = oracle_nvfp4(p, rows=rows)
    assert_close(bits(D[rows]), ref, T, "beyond 2^31: rows")
    _, T, ref = oracle_nvfp4(p, cols=cols)
    assert_close(bits(D[:, cols]), ref, T, "beyond 2^31: cols")
    del flat, D
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["nvfp4_4096", "nvfp4_16384"])
def test_nvfp4_full_size_sampled(dev, name):
    """Full-size workloads in the benchmark's launch configuration (default
    plan, nvfp4_gemm with row-major scales): sampled rows and columns."""
    w = workloads.WORKLOADS[name]
    p = workloads.make_nvfp4(w, dev)
    M, N, K = w.M, w.N, w.K
    flat, D = new_out(M, N, dev)
    bsg.nvfp4_gemm(M, N, K, p["A"], p["sfA"], p["B"], p["sfB"], p["alpha"], D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert_guard(flat)
    rows, cols = tile_samples(M, N, 128, 256, seed=M)
    if M > 8192:   # keep the oracle's share to seconds: every other M tile
        rows = rows[::2] + [M - 1]
    check_sampled_nvfp4(p, D, sorted(set(rows)), cols, name)


@pytest.mark.parametrize("name", [n for n in workloads.WORKLOADS if "skinny" in n])
def test_nvfp4_skinny_cells(dev, name):
    """The skinny-M weight GEMM cells, full comparison."""
    w = workloads.WORKLOADS[name]
    p = workloads.make_nvfp4(w, dev)
    got = gpu_nvfp4(p, dev)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, name)


# activation rows each skinny plan serves: one block of its tile, or two
# blocks where the tile is whole 128-row scale blocks
SKINNY_PLANS = {"nvfp4_skinny_m64_s3": 64, "nvfp4_skinny_m64_s6": 64, "nvfp4_skinny_m128_s3": 256,
                "nvfp4_skinny_m256_s4": 512}


@pytest.mark.parametrize("plan", list(SKINNY_PLANS))
@pytest.mark.parametrize("M,N,K", [(1, 136, 256), (16, 256, 512), (48, 1024, 1024), (37, 392, 1280),
                                   (64, 3072, 3072), (100, 1000, 2304), (256, 520, 4096), (200, 8, 512),
                                   (64, 16384, 512), (300, 264, 1536), (512, 392, 1024)])
def test_nvfp4_skinny_kernel(dev, plan, M, N, K):
    """The swap-AB split-K kernel forced on every shape it can serve: ragged
    M and N, the split chosen per call (cluster sizes from 1 to 8, some not
    dividing the k-blocks evenly), a wide N whose split is capped by
    residency, and two activation blocks (M past the plan's tile)."""
    if M > SKINNY_PLANS[plan]:
        pytest.skip("activation rows exceed the plan's tile")
    bsg.bsg_force_plan(plan)
    try:
        p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
        got = gpu_nvfp4(p, dev)
    finally:
        bsg.bsg_force_plan(None)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, f"{plan} {M}x{N}x{K}")


# ---------------------------------------------------------------------------
# FP8
# ---------------------------------------------------------------------------

def gpu_fp8(q, dev, sA=None, sB=None, alpha=None):
    M, N, K = q["M"], q["N"], q["K"]
    A, B = q["A"].to(dev), q["B"].to(dev)
    flat, D = new_out(M, N, dev)
    ta = None if sA is None else torch.tensor([sA], dtype=torch.float32, device=dev)
    tb = None if sB is None else torch.tensor([sB], dtype=torch.float32, device=dev)
    bsg.fp8_gemm(M, N, K, A, ta, B, tb, q["alpha"] if alpha is None else alpha, D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert_guard(flat)
    return bits(D)


@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (200, 136, 384), (1, 8, 128), (300, 520, 1024)])
def test_fp8_parity(dev, fp8_plan, M, N, K):
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=M, N=N, K=K)
    got = gpu_fp8(q, dev)
    _, T, ref = oracle.get().fp8_gemm(q["A"].numpy(), q["B"].numpy(), q["alpha"])
    assert_close(got, ref, T, f"fp8 {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(256, 512, 512), (300, 768, 1024), (520, 1024, 2048), (1, 512, 128)])
def test_fp8_wide_pair_plan(dev, M, N, K):
    """The 512-wide FP8 pair plan (each CTA's 128 rows of both 256-row B
    halves in one 3-D copy, two N = 256 MMAs per K step into one accumulator
    that fills TMEM): oracle parity, and bit for bit the 256-wide pair plan,
    since every output accumulates over K in the same order. N = 768 leaves
    the second tile's upper half past N (zero-filled, not stored)."""
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=M, N=N, K=K)
    got = {}
    for plan in ("fp8_tc2_256x512_s4_acc1", "fp8_tc2_256x256_s6_acc2"):
        bsg.bsg_force_plan(plan)
        try:
            got[plan] = gpu_fp8(q, dev)
            assert bsg.bsg_last_plan_name() == plan
        finally:
            bsg.bsg_force_plan(None)
    assert np.array_equal(got["fp8_tc2_256x512_s4_acc1"], got["fp8_tc2_256x256_s6_acc2"])
    _, T, ref = oracle.get().fp8_gemm(q["A"].numpy(), q["B"].numpy(), q["alpha"])
    assert_close(got["fp8_tc2_256x512_s4_acc1"], ref, T, f"fp8 wide {M}x{N}x{K}")


def test_fp8_wide_pair_plan_needs_whole_halves(dev):
    """Forced with N not a multiple of 256, the 512-wide plan (whose B view
    tiles N in 256-row halves) is refused before any launch."""
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=256, N=520, K=256)
    flat, D = new_out(256, 520, dev)
    bsg.bsg_force_plan("fp8_tc2_256x512_s4_acc1")
    try:
        rc = bsg.load().fp8_gemm(256, 520, 256, q["A"].to(dev).data_ptr(), None, q["B"].to(dev).data_ptr(), None,
                                 q["alpha"], D.data_ptr(), None)
    finally:
        bsg.bsg_force_plan(None)
    assert rc == bsg.BSG_ERR_NO_PLAN
    assert bsg.bsg_last_launch_count() == 0


def test_fp8_device_scales(dev):
    """alpha * sA * sB with sA, sB read from device memory."""
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=256, N=384, K=512)
    got = gpu_fp8(q, dev, sA=0.375, sB=-2.5, alpha=1.25)
    _, T, ref = oracle.get().fp8_gemm(q["A"].numpy(), q["B"].numpy(), 1.25, 0.375, -2.5)
    assert_close(got, ref, T, "fp8 device scales")


def test_fp8_full_size_sampled(dev):
    w = workloads.WORKLOADS["fp8_8192"]
    q = workloads.make_fp8(w, dev)
    M, N, K = w.M, w.N, w.K
    flat, D = new_out(M, N, dev)
    bsg.fp8_gemm(M, N, K, q["A"], None, q["B"], None, q["alpha"], D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert_guard(flat)
    rows, cols = tile_samples(M, N, 128, 256, seed=3)
    Dh = bits(D)
    A, B = q["A"].cpu().numpy(), q["B"].cpu().numpy()
    _, T, ref = oracle.get().fp8_gemm(A, B, q["alpha"], rows=rows)
    assert_close(Dh[rows], ref, T, "fp8 8192 rows")
    _, T, ref = oracle.get().fp8_gemm(A, B, q["alpha"], cols=cols)
    assert_close(Dh[:, cols], ref, T, "fp8 8192 cols")


@pytest.mark.parametrize("splits", [1, 2, 3, 4, 5, 6, 8])
@pytest.mark.parametrize("plan,M", [("nvfp4_skinny_m64_s3", 64), ("nvfp4_skinny_m64_s6", 40),
                                    ("nvfp4_skinny_m128_s3", 200), ("nvfp4_skinny_m256_s4", 384)])
def test_nvfp4_skinny_every_split(dev, plan, M, splits):
    """Every cluster size the kernel takes, forced: weight rows owned in 8-row
    groups, unevenly for 3, 5 and 6 splits; k-blocks (18) split unevenly for
    4, 5 and 8; two activation blocks for the m128 and m256 plans."""
    N, K = 392, 4608
    if plan == "nvfp4_skinny_m256_s4" and splits == 5:
        pytest.skip("the m256 plan's receive area holds no five-way split")
    bsg.bsg_force_plan(plan)
    bsg.bsg_set_skinny_splits(splits)
    try:
        p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
        got = gpu_nvfp4(p, dev)
    finally:
        bsg.bsg_set_skinny_splits(0)
        bsg.bsg_force_plan(None)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, f"{plan} S={splits} {M}x{N}x{K}")


# ---------------------------------------------------------------------------
# Runtime behaviour
# ---------------------------------------------------------------------------

def test_watchdog_reports_timeout_and_context_survives(dev):
    """A bounded wait on a barrier nothing arrives on ends with a status code,
    not a hang; the context stays usable for the next GEMM."""
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    bsg.bsg_watchdog_selftest(20_000_000)          # 20 ms
    assert bsg.bsg_get_device_status() == bsg.BSG_ERR_DEVICE_TIMEOUT
    assert bsg.bsg_last_status_word() == (bsg.BSG_ERR_DEVICE_TIMEOUT << 16) | 0xF
    assert bsg.bsg_get_device_status() == bsg.BSG_OK   # reading clears it
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_256"], "cpu")
    got = gpu_nvfp4(p, dev)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, "nvfp4 after watchdog")


def test_stream_ordering(dev):
    """Calls on a side stream are ordered on that stream."""
    s = torch.cuda.Stream()
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=256, N=256, K=512)
    with torch.cuda.stream(s):
        got = gpu_nvfp4(p, dev, "swizzled", stream=s)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, "side stream")


# ---------------------------------------------------------------------------
# Replicas: a GEMM split by output columns into per-rank calls
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("world", [2, 3])
def test_column_shards_concatenate(dev, world):
    """The calls a column-split job makes, run one after another on this GPU:
    rank r multiplies A by its rows [n0, n1) of B (with those rows' scales)
    into its own [M, n1 - n0] block; the blocks, concatenated, match the
    unsharded oracle result."""
    from block_scaled_precision_persistent_gb300.replicas import shard_range
    M, N, K = 300, 648, 1024
    p = workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)
    A, sfA = p["A"].to(dev), p["sfA"].to(dev)
    blocks = []
    for r in range(world):
        n0, n1 = shard_range(N, world, r)
        B = p["B"][n0:n1].contiguous().to(dev)
        sfB = p["sfB"][n0:n1].contiguous().to(dev)
        flat, D = new_out(M, n1 - n0, dev)
        bsg.nvfp4_gemm(M, n1 - n0, K, A, sfA, B, sfB, p["alpha"], D)
        torch.cuda.synchronize()
        assert bsg.bsg_get_device_status() == bsg.BSG_OK
        assert_guard(flat)
        blocks.append(bits(D))
    got = np.concatenate(blocks, axis=1)
    _, T, ref = oracle_nvfp4(p)
    assert_close(got, ref, T, f"{world} column shards")
