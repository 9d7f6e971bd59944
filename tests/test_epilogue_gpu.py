"""GPU parity of the fused epilogue variants against the CPU oracle.

D[scatter[m]][n] = bf16(gamma[m] * (alpha * acc[m][n] + bias[n])), the shared
bias, per-row gamma and scattered output rows of "Triton #11171 - Why Two New
NVFP4 Test Cases Produced Twelve Tensor-Memory Failures". Every compiled
plan (1-SM, CTA pair, skinny split-K; NVFP4 and FP8) is forced on ragged
shapes that span several tiles, with each option alone and all together.
Rows of D that no scatter index names must keep their prefill bit for bit;
written rows are compared element by element under the GEMM tolerance with
T' = |gamma| (T + |bias|). The hand-worked case of
tests/golden/nvfp4_epilogue_case.txt is checked exactly, and the full
16384^3 workload, in the benchmark's launch configuration, on sampled rows
and columns.
"""
from __future__ import annotations

from pathlib import Path

import numpy as np
import pytest
import torch

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg
import oracle
import workloads

pytestmark = pytest.mark.gpu

GOLDEN = Path(__file__).resolve().parent / "golden"
SENTINEL = 0x7FC1          # a NaN pattern no computed output can have
GUARD = 256

NVFP4_PLANS = ["nvfp4_tc1_128x256_s3_acc1", "nvfp4_tc1_128x128_s5_acc2",
               "nvfp4_tc2_256x256_s5_acc1", "nvfp4_tc2_256x128_s6_acc2"]
SKINNY_PLANS = {"nvfp4_skinny_m64_s3": 64, "nvfp4_skinny_m64_s6": 64, "nvfp4_skinny_m128_s3": 256,
                "nvfp4_skinny_m256_s4": 512}
FP8_PLANS = ["fp8_tc1_128x256_s4_acc2", "fp8_tc1_128x128_s6_acc2", "fp8_tc2_256x256_s6_acc2"]
VARIANTS = ["bias", "gamma", "bias_gamma", "scatter", "all", "all_drop"]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    bsg.bsg_force_plan(None)
    return d


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def variant_inputs(variant: str, M: int, N: int, seed: int, bias_std: float):
    """(bias, gamma, scatter, m_out) on the CPU for one variant; scattered
    variants write into a D with more rows than M (rows left untouched)."""
    drop = 0.25 if variant == "all_drop" else 0.0
    m_out = M + 37 if variant in ("scatter", "all", "all_drop") else M
    e = workloads.make_epilogue(M, N, seed, m_out=m_out, drop=drop, bias_std=bias_std)
    if variant == "all_drop" and M > 2:
        e["scatter"][1] = m_out + 5            # out of range: not written either
    return (e["bias"] if "bias" in variant or variant.startswith("all") else None,
            e["gamma"] if "gamma" in variant or variant.startswith("all") else None,
            e["scatter"] if variant in ("scatter", "all", "all_drop") else None, m_out)


def run_gpu(kind, p, dev, bias, gamma, scatter, m_out):
    """One _ex call; D prefilled with SENTINEL plus a guard tail. Returns D bits."""
    M, N, K = p["M"], p["N"], p["K"]
    flat = torch.full((m_out * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    D = flat[: m_out * N].view(torch.bfloat16).view(m_out, N)
    dv = lambda t: None if t is None else t.to(dev)  # noqa: E731
    if kind == "nvfp4":
        A, B = p["A"].to(dev), p["B"].to(dev)
        sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
        sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
        bsg.nvfp4_swizzle_scales(M, K, p["sfA"].to(dev), sa)
        bsg.nvfp4_swizzle_scales(N, K, p["sfB"].to(dev), sb)
        bsg.nvfp4_gemm_ex(M, N, K, A, sa, B, sb, p["alpha"], dv(bias), dv(gamma), dv(scatter), m_out, D)
    else:
        bsg.fp8_gemm_ex(M, N, K, p["A"].to(dev), None, p["B"].to(dev), None, p["alpha"], dv(bias),
                        dv(gamma), dv(scatter), m_out, D)
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert (bits(flat[-GUARD:]) == SENTINEL).all(), "kernel wrote past the end of D"
    return bits(D)


def oracle_ref(kind, p, bias, gamma, rows=None, cols=None):
    npy = lambda t: None if t is None else t.numpy()  # noqa: E731
    o = oracle.get()
    if kind == "nvfp4":
        return o.nvfp4_gemm(p["A"].cpu().numpy(), p["sfA"].cpu().numpy(), p["B"].cpu().numpy(),
                            p["sfB"].cpu().numpy(), p["alpha"], p["K"], rows=rows, cols=cols,
                            bias=npy(bias), gamma=npy(gamma))
    return o.fp8_gemm(p["A"].cpu().numpy(), p["B"].cpu().numpy(), p["alpha"], rows=rows, cols=cols,
                      bias=npy(bias), gamma=npy(gamma))


def check(got, kind, p, bias, gamma, scatter, m_out, what):
    """Written rows within tolerance of the oracle; every other row of D
    still holds the prefill."""
    _, T, ref = oracle_ref(kind, p, bias, gamma)
    if scatter is None:
        dst = np.arange(p["M"])
    else:
        dst = scatter.numpy().astype(np.int64)
    live = (dst >= 0) & (dst < m_out)
    ok = oracle.within_tolerance(got[dst[live]], ref[live], T[live])
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first at "
                             f"computed row {np.flatnonzero(live)[i]}, col {j}: gpu="
                             f"{oracle.bf16_bits_to_float(got[dst[live]][i, j])} ref="
                             f"{oracle.bf16_bits_to_float(ref[live][i, j])}")
    untouched = np.ones(m_out, bool)
    untouched[dst[live]] = False
    assert (got[untouched] == SENTINEL).all(), f"{what}: a row no index names was written"


def nvfp4_problem(M, N, K):
    return workloads.make_nvfp4(workloads.WORKLOADS["nvfp4_4096"], "cpu", M=M, N=N, K=K)


def out_std(K):
    """Typical |D| of the N(0,1) two-level workloads (sqrt K): the bias is
    drawn on that scale so that it matters and cancels now and then."""
    return float(np.sqrt(K))


@pytest.fixture
def forced(request, dev):
    yield
    bsg.bsg_force_plan(None)


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("plan", [None] + NVFP4_PLANS)
def test_nvfp4_epilogue_plans(dev, forced, plan, variant):
    """Ragged M and N over several 256 x 256 tiles, every 1-SM and pair plan."""
    M, N, K = 600, 712, 1280
    bsg.bsg_force_plan(plan)
    p = nvfp4_problem(M, N, K)
    bias, gamma, scatter, m_out = variant_inputs(variant, M, N, seed=11, bias_std=out_std(K))
    got = run_gpu("nvfp4", p, dev, bias, gamma, scatter, m_out)
    check(got, "nvfp4", p, bias, gamma, scatter, m_out, f"{plan} {variant}")


@pytest.mark.parametrize("variant", ["bias_gamma", "all_drop"])
@pytest.mark.parametrize("plan", list(SKINNY_PLANS))
@pytest.mark.parametrize("M,N,K", [(1, 136, 256), (37, 392, 1280), (64, 3072, 3072), (200, 520, 4096),
                                   (100, 1000, 2304), (400, 264, 3072)])
def test_nvfp4_epilogue_skinny(dev, forced, plan, M, N, K, variant):
    """The swap-AB split-K kernel (bias per weight row, gamma and scatter per
    activation row), over the splits chosen per call and two activation
    blocks."""
    if M > SKINNY_PLANS[plan]:
        pytest.skip("activation rows exceed the plan's tile")
    bsg.bsg_force_plan(plan)
    p = nvfp4_problem(M, N, K)
    bias, gamma, scatter, m_out = variant_inputs(variant, M, N, seed=M, bias_std=out_std(K))
    got = run_gpu("nvfp4", p, dev, bias, gamma, scatter, m_out)
    check(got, "nvfp4", p, bias, gamma, scatter, m_out, f"{plan} {M}x{N}x{K} {variant}")


@pytest.mark.parametrize("variant", ["bias_gamma", "all", "all_drop"])
@pytest.mark.parametrize("plan", [None] + FP8_PLANS)
def test_fp8_epilogue_plans(dev, forced, plan, variant):
    M, N, K = 300, 520, 1024
    bsg.bsg_force_plan(plan)
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=M, N=N, K=K)
    bias, gamma, scatter, m_out = variant_inputs(variant, M, N, seed=5, bias_std=out_std(K))
    got = run_gpu("fp8", q, dev, bias, gamma, scatter, m_out)
    check(got, "fp8", q, bias, gamma, scatter, m_out, f"{plan} {variant}")


@pytest.mark.parametrize("variant", ["bias_gamma", "all", "all_drop"])
def test_fp8_epilogue_wide_plan(dev, forced, variant):
    """The 512-wide FP8 pair plan (eight epilogue warps of 256 columns, one
    staging buffer each): N = 768 leaves the second tile's upper half past N."""
    M, N, K = 300, 768, 1024
    bsg.bsg_force_plan("fp8_tc2_256x512_s4_acc1")
    q = workloads.make_fp8(workloads.WORKLOADS["fp8_8192"], "cpu", M=M, N=N, K=K)
    bias, gamma, scatter, m_out = variant_inputs(variant, M, N, seed=7, bias_std=out_std(K))
    got = run_gpu("fp8", q, dev, bias, gamma, scatter, m_out)
    assert bsg.bsg_last_plan_name() == "fp8_tc2_256x512_s4_acc1"
    check(got, "fp8", q, bias, gamma, scatter, m_out, f"fp8 wide {variant}")


def test_epilogue_worked_case(dev):
    """tests/golden/nvfp4_epilogue_case.txt on the GPU, exactly: K padded
    from 16 to 256 with zero codes (the sums do not change) and N from 4 to
    8 with zero B rows and zero bias (columns 4..7 are not compared)."""
    g = {}
    for line in (GOLDEN / "nvfp4_epilogue_case.txt").read_text().splitlines():
        t = line.split()
        if t and not t[0].startswith("#"):
            g.setdefault(t[0], []).append(t[1:])
    K = 256
    ac = [int(c, 16) for c in g["acodes"][0]]
    bc = [int(c, 16) for c in g["bcodes"][0]] + [0] * 4
    codes = lambda cs: torch.tensor([[c] * 16 + [0] * (K - 16) for c in cs], dtype=torch.uint8)  # noqa: E731
    pk = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).contiguous()  # noqa: E731
    M, N = len(ac), len(bc)
    p = dict(M=M, N=N, K=K, A=pk(codes(ac)), B=pk(codes(bc)),
             sfA=torch.full((M, K // 16), 0x38, dtype=torch.uint8),
             sfB=torch.full((N, K // 16), 0x38, dtype=torch.uint8), alpha=float(g["alpha"][0][0]))
    bias = torch.tensor([float(v) for v in g["bias"][0]] + [0.0] * 4, dtype=torch.float32)
    gamma = torch.tensor([float(v) for v in g["gamma"][0]], dtype=torch.float32)
    scatter = torch.tensor([int(v) for v in g["scatter"][0]], dtype=torch.int32)
    got = oracle.bf16_bits_to_float(run_gpu("nvfp4", p, dev, bias, gamma, None, M))
    for r in g["D"]:
        want = [float(v) for v in r[1:]]
        assert got[int(r[0])][:4].tolist() == want, (r[0], got[int(r[0])])
        assert np.signbit(got[int(r[0])][:4]).tolist() == np.signbit(want).tolist(), r[0]
    got = oracle.bf16_bits_to_float(run_gpu("nvfp4", p, dev, bias, gamma, scatter, M))
    for r in g["out"]:
        want = np.array([float(v) for v in r[1:]])
        row = got[int(r[0])][:4]
        assert np.array_equal(np.isnan(row), np.isnan(want))
        assert np.array_equal(row[~np.isnan(want)], want[~np.isnan(want)]), r[0]


@pytest.mark.parametrize("plan", [None, "nvfp4_tc2_256x256_s5_acc1", "nvfp4_tc1_128x128_s5_acc2",
                                  "nvfp4_skinny_m128_s3"])
def test_identity_epilogue_matches_plain(dev, forced, plan):
    """bias = 0, gamma = 1 through the epilogue-variant kernels equals the
    plain kernels bit for bit (zeros compared without their sign)."""
    M, N, K = 96 if plan and "skinny" in plan else 520, 392, 2048
    bsg.bsg_force_plan(plan)
    p = nvfp4_problem(M, N, K)
    plain = run_gpu("nvfp4", p, dev, None, None, None, M)
    ex = run_gpu("nvfp4", p, dev, torch.zeros(N), torch.ones(M), None, M)
    nz = lambda b: np.where((b & 0x7FFF) == 0, 0, b)  # noqa: E731
    assert np.array_equal(nz(plain), nz(ex))


def test_full_size_all_variants_sampled(dev):
    """16384^3 in the benchmark's launch configuration (default plan) with
    bias, gamma and a scatter permutation: sampled computed rows (every
    256-row tile) and columns (every 256-column tile) against the oracle."""
    w = workloads.WORKLOADS["nvfp4_16384"]
    p = workloads.make_nvfp4(w, dev)
    M, N, K = w.M, w.N, w.K
    e = workloads.make_epilogue(M, N, seed=3, bias_std=out_std(K))
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"], sa)
    bsg.nvfp4_swizzle_scales(N, K, p["sfB"], sb)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    bsg.nvfp4_gemm_ex(M, N, K, p["A"], sa, p["B"], sb, p["alpha"], e["bias"].to(dev), e["gamma"].to(dev),
                      e["scatter"].to(dev), M, D)
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    cpu = {k: p[k].cpu() for k in ("A", "sfA", "B", "sfB")}
    cpu.update(M=M, N=N, K=K, alpha=p["alpha"])
    rng = np.random.default_rng(16384)
    rows = sorted({int(t * 256 + rng.integers(256)) for t in range(0, M // 256, 2)} | {M - 1})
    cols = sorted({int(t * 256 + rng.integers(256)) for t in range(N // 256)} | {N - 1})
    dst = e["scatter"].numpy().astype(np.int64)
    Dh = bits(D)
    _, T, ref = oracle_ref("nvfp4", cpu, e["bias"], e["gamma"], rows=rows)
    assert oracle.within_tolerance(Dh[dst[rows]], ref, T).all(), "sampled rows"
    crow = list(range(0, M, 97))
    _, T, ref = oracle_ref("nvfp4", cpu, e["bias"], e["gamma"], rows=crow, cols=cols)
    assert oracle.within_tolerance(Dh[np.ix_(dst[crow], cols)], ref, T).all(), "sampled cols"


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("M,N,K", [(300, 392, 768), (130, 120, 1280)])
def test_packed_plan_epilogue(dev, variant, M, N, K):
    """The tile-packed plan (nvfp4_gemm_packed_ex) with each epilogue variant;
    130 x 120 leaves the peer CTA's row blocks of A and B past M and N."""
    p = nvfp4_problem(M, N, K)
    bias, gamma, scatter, m_out = variant_inputs(variant, M, N, seed=M + N, bias_std=out_std(K))
    flat = torch.full((m_out * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    D = flat[: m_out * N].view(torch.bfloat16).view(m_out, N)
    dv = lambda t: None if t is None else t.to(dev)  # noqa: E731
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales2(M, N, K, p["sfA"].to(dev), sa, p["sfB"].to(dev), sb)
    ap = torch.empty(bsg.nvfp4_packed_operand_bytes(M, K), dtype=torch.uint8, device=dev)
    bp = torch.empty(bsg.nvfp4_packed_operand_bytes(N, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_pack_operand(M, K, p["A"].to(dev), ap)
    bsg.nvfp4_pack_operand(N, K, p["B"].to(dev), bp)
    bsg.nvfp4_gemm_packed_ex(M, N, K, ap, sa, bp, sb, p["alpha"], dv(bias), dv(gamma), dv(scatter), m_out, D)
    assert bsg.bsg_last_plan_name() == "nvfp4_tc2_256x256_s5_acc1_packed"
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert (bits(flat[-GUARD:]) == SENTINEL).all(), "kernel wrote past the end of D"
    check(bits(D), "nvfp4", p, bias, gamma, scatter, m_out, f"packed {variant} {M}x{N}x{K}")
