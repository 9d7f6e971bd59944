"""GPU parity of the inner-expert (K-ragged) NVFP4 x dense GEMM against the
CPU oracle, with BF16 and FP16 right-hand sides.

"Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
Failures", section "Why `pad_a` represents the K-ragged boundary": the
ragged dimension is A's K, padded per slice, and each slice of K gives its
own output. Ragged K splits (empty slices, one-block slices, one slice over
all of K), M not a multiple of 128 (so slice outputs abut inside a tile),
bias per slice and gamma, both TMEM-staged plans, the hand-worked case of
tests/golden/nvfp4_dense_kragged_case.txt exactly, and a single slice bit
for bit against the plain dense GEMM.
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


def koffsets(blocks) -> torch.Tensor:
    """Slice sizes in 64-element blocks -> int32 offsets along K."""
    o = np.zeros(len(blocks) + 1, np.int32)
    o[1:] = np.cumsum(blocks) * 64
    return torch.from_numpy(o)


def gpu_kragged(p, koffs, dev, bias=None, gamma=None):
    M, N, K = p["M"], p["N"], p["K"]
    E = koffs.numel() - 1
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"].to(dev), sa)
    flat = torch.full((E * M * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    D = flat[: E * M * N].view(torch.bfloat16).view(E, M, N)
    dv = lambda t: None if t is None else t.to(dev)  # noqa: E731
    call = bsg.nvfp4_dense_f16_kgrouped_gemm if p["B"].dtype == torch.float16 else bsg.nvfp4_dense_kgrouped_gemm
    call(E, M, N, K, p["A"].to(dev), sa, p["B"].to(dev), koffs.to(dev), p["alpha"], dv(bias), dv(gamma), D)
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert (bits(flat[-GUARD:]) == SENTINEL).all(), "kernel wrote past the end of D"
    return bits(D)


def check(got, p, koffs, bias, gamma, what):
    npy = lambda t: None if t is None else t.cpu().numpy()  # noqa: E731
    _, T, ref = oracle.get().nvfp4_dense_kgrouped_gemm(p["A"].cpu().numpy(), p["sfA"].cpu().numpy(), bits(p["B"]),
                                                       koffs.numpy(), p["alpha"], p["K"], bias=npy(bias),
                                                       gamma=npy(gamma), b_f16=p["B"].dtype == torch.float16)
    E = ref.shape[0]
    for e in range(E):
        ok = oracle.within_tolerance(got[e], ref[e], T[e])
        if not ok.all():
            i, j = np.argwhere(~ok)[0]
            raise AssertionError(f"{what} slice {e}: {int((~ok).sum())} of {ok.size} outside tolerance; first at "
                                 f"({i},{j}): gpu={oracle.bf16_bits_to_float(got[e, i, j])} "
                                 f"ref={oracle.bf16_bits_to_float(ref[e, i, j])}")


SPLITS = {
    "one_slice": [20],
    "ragged": [3, 0, 1, 9, 2, 5],
    "empty_ends": [0, 0, 12, 8, 0],
    "single_blocks": [1] * 20,
}


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("split", list(SPLITS))
@pytest.mark.parametrize("plan", PLANS)
def test_kragged_splits(dev, forced, plan, split, b_dtype):
    koffs = koffsets(SPLITS[split])
    M, N, K = 200, 392, int(koffs[-1])
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense(M, N, K, seed=K + len(SPLITS[split]), b_dtype=b_dtype)
    got = gpu_kragged(p, koffs, dev)
    check(got, p, koffs, None, None, f"{plan} {split}")


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("plan", PLANS)
def test_kragged_bias_gamma(dev, forced, plan, b_dtype):
    """A bias row per slice and gamma per row, with an empty slice (whose
    output is gamma * bias) and M = 300 (slice outputs abut mid-tile)."""
    koffs = koffsets([4, 0, 7, 5])
    E, M, N, K = 4, 300, 520, int(koffs[-1])
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense(M, N, K, seed=9, b_dtype=b_dtype)
    rng = np.random.default_rng(6)
    bias = torch.from_numpy((rng.standard_normal((E, N)) * 8).astype(np.float32))
    gamma = torch.from_numpy((1 + 0.5 * rng.standard_normal(M)).astype(np.float32))
    got = gpu_kragged(p, koffs, dev, bias, gamma)
    check(got, p, koffs, bias, gamma, f"{plan} bias gamma")


def test_kragged_worked_case(dev):
    """tests/golden/nvfp4_dense_kragged_case.txt exactly. The slices are
    padded from 16 to 64 elements (zero codes in A, zeros in B) and N from 2
    to 8, so koffs = 0, 64, 128."""
    want = {}
    for line in (GOLDEN / "nvfp4_dense_kragged_case.txt").read_text().splitlines():
        t = line.split()
        if t and t[0] == "D":
            want[(int(t[1]), int(t[2]))] = [float(v) for v in t[3:]]
    K, N = 128, 8
    codes = np.zeros((2, K), np.uint8)
    codes[0, 0:16] = codes[0, 64:80] = 0x2
    codes[1, 0:16] = codes[1, 64:80] = [k % 8 for k in range(16)]
    A = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))
    sfA = torch.full((2, K // 16), 0x38, dtype=torch.uint8)
    sfA[0, 0], sfA[0, 4] = 0x40, 0x30                   # block scales 2.0 and 0.5 of row 0
    B = torch.zeros((N, K), dtype=torch.bfloat16)
    B[0, 0:16], B[0, 64:80], B[1, 0:16], B[1, 64:80] = 0.25, -3.0, 1.5, 1.5
    bias = torch.zeros((2, N), dtype=torch.float32)
    bias[1, 0] = 100.0
    p = dict(M=2, N=N, K=K, A=A, sfA=sfA, B=B, alpha=1.0)
    got = oracle.bf16_bits_to_float(gpu_kragged(p, koffsets([1, 1]), dev, bias))
    for (e, i), row in want.items():
        assert got[e, i, :2].tolist() == row, (e, i, got[e, i, :2])


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("plan", PLANS[1:])
def test_kragged_single_slice_matches_plain(dev, forced, plan, b_dtype):
    """One slice over all of K: the K-ragged kernel equals the plain dense
    kernel of the same plan bit for bit (zeros compared without sign)."""
    M, N, K = 520, 392, 2048
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense(M, N, K, seed=13, b_dtype=b_dtype)
    got = gpu_kragged(p, torch.tensor([0, K], dtype=torch.int32), dev)[0]
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"].to(dev), sa)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    plain = bsg.nvfp4_dense_f16_gemm if b_dtype == torch.float16 else bsg.nvfp4_dense_gemm
    plain(M, N, K, p["A"].to(dev), sa, p["B"].to(dev), p["alpha"], None, None, None, M, D)
    torch.cuda.synchronize()
    nz = lambda b: np.where((b & 0x7FFF) == 0, 0, b)  # noqa: E731
    assert np.array_equal(nz(got), nz(bits(D)))
