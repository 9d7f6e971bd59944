"""GPU parity of the grouped (routed) NVFP4 x dense GEMM against the CPU
oracle, with BF16 and FP16 right-hand sides.

"Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
Failures", section "Ragged mode added routing rather than a plain matrix",
with the dense operand of its opening: routed rows form slices, each
multiplied by its own dense right-hand side, under the routed, scatter and
gamma variants. Ragged splits (empty slices, slices of a few rows, slices
ending inside a warp's rows or crossing 128-row tiles), both TMEM-staged
plans, the epilogue variants with the scatter back to token order, the
hand-worked case of tests/golden/nvfp4_dense_grouped_case.txt exactly, one
slice against the plain dense GEMM bit for bit, and whole slices of the MoE
workload (64 experts, 1024 tokens x top-8, 4096 x 7168).
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
SENTINEL = 0x7FC1
GUARD = 256
PLANS = [None, "nvfp4bf16_tc1_128x128_s8_acc2_tmema", "nvfp4bf16_tc1_128x256_s5_acc1_tmema"]
DTYPES = [torch.bfloat16, torch.float16]


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    d = torch.device("cuda:0")
    torch.cuda.set_device(d)
    bsg.bsg_force_plan(None)
    return d


@pytest.fixture
def forced(dev):
    yield
    bsg.bsg_force_plan(None)


def bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def offsets(sizes) -> torch.Tensor:
    o = np.zeros(len(sizes) + 1, np.int32)
    o[1:] = np.cumsum(sizes)
    return torch.from_numpy(o)


def gpu_dense_grouped(p, offs, dev, bias=None, gamma=None, scatter=None, m_out=None):
    E, M, N, K = p["E"], p["M"], p["N"], p["K"]
    m_out = M if m_out is None else m_out
    sa = torch.empty(bsg.nvfp4_grouped_scale_bytes(E, M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales_grouped(E, M, K, offs.to(dev), p["sfA"].to(dev), sa)
    flat = torch.full((m_out * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    D = flat[: m_out * N].view(torch.bfloat16).view(m_out, N)
    dv = lambda t: None if t is None else t.to(dev)  # noqa: E731
    call = bsg.nvfp4_dense_f16_grouped_gemm if p["B"].dtype == torch.float16 else bsg.nvfp4_dense_grouped_gemm
    call(E, M, N, K, p["A"].to(dev), sa, p["B"].to(dev), offs.to(dev), p["alpha"], dv(bias), dv(gamma),
         dv(scatter), m_out, D)
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert (bits(flat[-GUARD:]) == SENTINEL).all(), "kernel wrote past the end of D"
    return bits(D)


def oracle_dense_grouped(p, offs, bias=None, gamma=None):
    npy = lambda t: None if t is None else t.cpu().numpy()  # noqa: E731
    return oracle.get().nvfp4_dense_grouped_gemm(p["A"].cpu().numpy(), p["sfA"].cpu().numpy(), bits(p["B"]),
                                                 offs.numpy(), p["alpha"], p["K"], bias=npy(bias),
                                                 gamma=npy(gamma), b_f16=p["B"].dtype == torch.float16)


def check(got, p, offs, bias, gamma, scatter, m_out, what):
    _, T, ref = oracle_dense_grouped(p, offs, bias, gamma)
    M = p["M"]
    dst = np.arange(M) if scatter is None else scatter.numpy().astype(np.int64)
    live = (dst >= 0) & (dst < m_out)
    ok = oracle.within_tolerance(got[dst[live]], ref[live], T[live])
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        r = np.flatnonzero(live)[i]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first at row {r} "
                             f"col {j}: gpu={oracle.bf16_bits_to_float(got[dst[r], j])} "
                             f"ref={oracle.bf16_bits_to_float(ref[r, j])}")
    untouched = np.ones(m_out, bool)
    untouched[dst[live]] = False
    assert (got[untouched] == SENTINEL).all(), f"{what}: a row no index names was written"


SPLITS = {
    "one_slice": [300],
    "ragged": [7, 0, 130, 1, 33, 129, 0, 64],
    "tiny": [1, 2, 3, 4, 5, 31, 32, 33],
    "empty_ends": [0, 0, 200, 56, 0],
}


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("split", list(SPLITS))
@pytest.mark.parametrize("plan", PLANS)
def test_dense_grouped_splits(dev, forced, plan, split, b_dtype):
    sizes = SPLITS[split]
    offs = offsets(sizes)
    E, M, N, K = len(sizes), int(offs[-1]), 392, 1280
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense_grouped(E, M, N, K, seed=len(sizes) + M, b_dtype=b_dtype)
    got = gpu_dense_grouped(p, offs, dev)
    check(got, p, offs, None, None, None, M, f"{plan} {split}")


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("plan", PLANS)
def test_dense_grouped_epilogue(dev, forced, plan, b_dtype):
    """A bias per slice, gamma per row, and the scatter back to token order
    of a top-3 routing of 100 tokens over 6 experts into a D with spare rows."""
    offs, dst = workloads.routing(6, 100, 3, seed=5)
    E, M, N, K = 6, 300, 520, 1024
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense_grouped(E, M, N, K, seed=7, b_dtype=b_dtype)
    rng = np.random.default_rng(3)
    bias = torch.from_numpy((rng.standard_normal((E, N)) * np.sqrt(K)).astype(np.float32))
    gamma = torch.from_numpy((1 + 0.5 * rng.standard_normal(M)).astype(np.float32))
    got = gpu_dense_grouped(p, offs, dev, bias, gamma, dst, M + 11)
    check(got, p, offs, bias, gamma, dst, M + 11, f"{plan} epilogue")


def test_dense_grouped_worked_case(dev):
    """tests/golden/nvfp4_dense_grouped_case.txt exactly (K padded 32 -> 64
    with zero codes, N 2 -> 8 with zero B rows and zero bias)."""
    want = {}
    for line in (GOLDEN / "nvfp4_dense_grouped_case.txt").read_text().splitlines():
        t = line.split()
        if t and t[0] == "D":
            want[int(t[1])] = [float(v) for v in t[2:]]
    K, N = 64, 8
    codes = np.zeros((3, K), np.uint8)
    codes[0, :32] = codes[2, :32] = 0x2
    codes[1, :32] = [k % 8 for k in range(32)]
    A = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))
    sfA = torch.tensor([[0x40, 0x30, 0x38, 0x38], [0x38, 0x38, 0x38, 0x38], [0x40, 0x30, 0x38, 0x38]],
                       dtype=torch.uint8)
    b0 = torch.zeros((N, K), dtype=torch.bfloat16)
    b0[0, :16], b0[0, 16:32], b0[1, :32] = 0.25, -3.0, 1.5
    b1 = b0.clone()
    b1[0], b1[1] = b0[1], b0[0]
    B = torch.stack([b0, b1])
    bias = torch.zeros((2, N), dtype=torch.float32)
    bias[0, :2] = torch.tensor([1.0, 2.0])
    bias[1, :2] = torch.tensor([10.0, 20.0])
    p = dict(E=2, M=3, N=N, K=K, A=A, sfA=sfA, B=B, alpha=1.0)
    got = oracle.bf16_bits_to_float(gpu_dense_grouped(p, torch.tensor([0, 2, 3], dtype=torch.int32), dev, bias))
    for i, row in want.items():
        assert got[i, :2].tolist() == row, (i, got[i, :2])


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("plan", PLANS[1:])
def test_dense_single_slice_matches_plain(dev, forced, plan, b_dtype):
    """One slice over every row: the grouped kernel equals the plain dense
    kernel of the same plan bit for bit (zeros compared without sign)."""
    M, N, K = 520, 392, 2048
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense_grouped(1, M, N, K, seed=12, b_dtype=b_dtype)
    got = gpu_dense_grouped(p, torch.tensor([0, M], dtype=torch.int32), dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"].to(dev), sa)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    plain = bsg.nvfp4_dense_f16_gemm if b_dtype == torch.float16 else bsg.nvfp4_dense_gemm
    plain(M, N, K, p["A"].to(dev), sa, p["B"][0].to(dev).contiguous(), p["alpha"], None, None, None, M, D)
    torch.cuda.synchronize()
    nz = lambda b: np.where((b & 0x7FFF) == 0, 0, b)  # noqa: E731
    assert np.array_equal(nz(got), nz(bits(D)))


def test_dense_grouped_rejects_other_plans(dev, forced):
    """A forced plan the grouped dense GEMM cannot run (A staged in shared
    memory) is refused before launch."""
    offs = offsets([64, 64])
    p = workloads.make_dense_grouped(2, 128, 64, 256, seed=1)
    sa = torch.empty(bsg.nvfp4_grouped_scale_bytes(2, 128, 256), dtype=torch.uint8, device=dev)
    D = torch.empty((128, 64), dtype=torch.bfloat16, device=dev)
    A, B, od = p["A"].to(dev), p["B"].to(dev), offs.to(dev)
    bsg.bsg_force_plan("nvfp4bf16_tc1_128x256_s3_acc2")
    rc = bsg.load().nvfp4_dense_grouped_gemm(2, 128, 64, 256, A.data_ptr(), sa.data_ptr(), B.data_ptr(),
                                             od.data_ptr(), 1.0, None, None, None, 128, D.data_ptr(), None)
    assert rc == bsg.BSG_ERR_NO_PLAN


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
def test_dense_grouped_moe_slices(dev, b_dtype):
    """The MoE workload with 16-bit expert weights (64 x 4096 x 7168) in the
    default plan: three whole slices (first, middle, last expert) against
    the oracle, with the bias per expert."""
    g = workloads.GROUPED_WORKLOADS["moe_e64_t1024_k8"]
    offs, _ = workloads.routing(g.E, g.tokens, g.top_k, seed=1)
    M = int(offs[-1])
    p = workloads.make_dense_grouped(g.E, M, g.N, g.K, seed=21, device=dev, b_dtype=b_dtype)
    bias = torch.from_numpy(np.random.default_rng(5).standard_normal((g.E, g.N)).astype(np.float32))
    got = gpu_dense_grouped(p, offs, dev, bias)
    o = oracle.get()
    A, sfA, B = p["A"].cpu().numpy(), p["sfA"].cpu().numpy(), p["B"]
    for e in (0, g.E // 2, g.E - 1):
        r0, r1 = int(offs[e]), int(offs[e + 1])
        if r1 == r0:
            continue
        _, T, ref = o.nvfp4_dense_gemm(A[r0:r1], sfA[r0:r1], bits(B[e]), p["alpha"], g.K, bias=bias[e].numpy(),
                                       b_f16=b_dtype == torch.float16)
        ok = oracle.within_tolerance(got[r0:r1], ref, T)
        assert ok.all(), (e, int((~ok).sum()))
