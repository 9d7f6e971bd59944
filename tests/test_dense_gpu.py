"""GPU parity of the NVFP4 x dense-BF16 and dense-FP16 GEMMs against the
CPU oracle.

"Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
Failures", opening: an NVFP4-scaled activation times a dense BF16 or FP16
operand. The kernel expands A to B's type (in shared or tensor memory) and
runs the 16-bit tensor core. One-hot probes check the expansion bit for bit
(every code, both nibbles, every swizzle row); shapes span several tiles with
ragged M, N and K, every dense plan, the pages' N = 256 case, and the
epilogue variants; the hand-worked cases of tests/golden/nvfp4_dense_case.txt
and nvfp4_dense_f16_case.txt are exact; 4096^3 is compared on sampled rows
and columns.
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

SENTINEL = 0x7FC1
GUARD = 256
PLANS = [None, "nvfp4bf16_tc1_128x128_s5_acc2", "nvfp4bf16_tc1_128x256_s3_acc2",
         "nvfp4bf16_tc1_128x256_s5_acc1_tmema", "nvfp4bf16_tc1_128x128_s8_acc2_tmema",
         "nvfp4bf16_tc2_256x256_s8_acc1_tmema"]


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


def gpu_dense(p, dev, bias=None, gamma=None, scatter=None, m_out=None):
    M, N, K = p["M"], p["N"], p["K"]
    m_out = M if m_out is None else m_out
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"].to(dev), sa)
    flat = torch.full((m_out * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    D = flat[: m_out * N].view(torch.bfloat16).view(m_out, N)
    dv = lambda t: None if t is None else t.to(dev)  # noqa: E731
    call = bsg.nvfp4_dense_f16_gemm if p["B"].dtype == torch.float16 else bsg.nvfp4_dense_gemm
    call(M, N, K, p["A"].to(dev), sa, p["B"].to(dev), p["alpha"], dv(bias), dv(gamma), dv(scatter), m_out, D)
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert (bits(flat[-GUARD:]) == SENTINEL).all(), "kernel wrote past the end of D"
    return bits(D)


def oracle_dense(p, rows=None, cols=None, bias=None, gamma=None):
    npy = lambda t: None if t is None else t.cpu().numpy()  # noqa: E731
    return oracle.get().nvfp4_dense_gemm(p["A"].cpu().numpy(), p["sfA"].cpu().numpy(), bits(p["B"]), p["alpha"],
                                         p["K"], rows=rows, cols=cols, bias=npy(bias), gamma=npy(gamma),
                                         b_f16=p["B"].dtype == torch.float16)


def assert_close(got, ref, T, what):
    ok = oracle.within_tolerance(got, ref, T)
    if not ok.all():
        i, j = np.argwhere(~ok)[0]
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} outside tolerance; first at ({i},{j}) "
                             f"gpu={oracle.bf16_bits_to_float(got[i, j])} ref={oracle.bf16_bits_to_float(ref[i, j])}")


DTYPES = [torch.bfloat16, torch.float16]


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("plan", PLANS)
@pytest.mark.parametrize("M,N,K", [(256, 256, 256), (1, 8, 64), (300, 392, 1280), (129, 520, 576),
                                   (600, 712, 2048)])
def test_dense_parity(dev, forced, plan, M, N, K, b_dtype):
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense(M, N, K, seed=M + N, b_dtype=b_dtype)
    got = gpu_dense(p, dev)
    _, T, ref = oracle_dense(p)
    assert_close(got, ref, T, f"{plan} {M}x{N}x{K}")


@pytest.mark.parametrize("plan", PLANS)
def test_dense_one_hot_expansion(dev, forced, plan):
    """A[i][k] = 1.0 (code 2, scale 1.0) only at k = pi(i): D[i][j] is then
    exactly B[j][pi(i)]. pi visits even and odd k, every 16-block and every
    64-element stage; rows cover every swizzle phase r % 8. With FP16 B, D is
    that value rounded to BF16: the oracle's result, bit for bit."""
    M, N, K = 256, 136, 512
    rng = np.random.default_rng(5)
    pi = rng.integers(0, K, M)
    codes = np.zeros((M, K), np.uint8)
    codes[np.arange(M), pi] = 0x2
    A = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))
    B = workloads.normal_bf16(N, K, 99, 1.0, "cpu").to(torch.bfloat16)
    p = dict(M=M, N=N, K=K, A=A, sfA=torch.full((M, K // 16), 0x38, dtype=torch.uint8), B=B, alpha=1.0)
    bsg.bsg_force_plan(plan)
    got = gpu_dense(p, dev)
    want = bits(B)[:, pi].T
    assert np.array_equal(got, want)
    # FP16 B with values BF16 cannot hold (11 significant bits)
    p["B"] = workloads.make_dense(8, N, K, seed=77, b_dtype=torch.float16)["B"] * 3.0
    got = gpu_dense(p, dev)
    _, _, ref = oracle_dense(p)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
def test_dense_scale_and_sign_probe(dev, b_dtype):
    """Every E2M1 code times a spread of E4M3 scales (subnormal to 448),
    against one-hot B rows: D[i][j] = e2m1(code) * scale exactly."""
    K, N = 64, 64
    codes = np.arange(16, dtype=np.uint8)
    scales = np.array([0x01, 0x07, 0x08, 0x30, 0x38, 0x41, 0x6F, 0x7E], np.uint8)
    M = codes.size * scales.size
    A_codes = np.zeros((M, K), np.uint8)
    sfA = np.full((M, K // 16), 0x38, np.uint8)
    for i, (c, s) in enumerate((c, s) for c in codes for s in scales):
        A_codes[i, :] = c
        sfA[i, :] = s
    A = torch.from_numpy((A_codes[:, 0::2] | (A_codes[:, 1::2] << 4)).astype(np.uint8))
    B = torch.zeros((N, K), dtype=b_dtype)
    B[torch.arange(N), torch.arange(N) % K] = 1.0          # B row j one-hot at k = j
    p = dict(M=M, N=N, K=K, A=A, sfA=torch.from_numpy(sfA), B=B, alpha=1.0)
    got = gpu_dense(p, dev)
    _, T, ref = oracle_dense(p)
    assert np.array_equal(np.where((got & 0x7FFF) == 0, 0, got), np.where((ref & 0x7FFF) == 0, 0, ref))


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
@pytest.mark.parametrize("plan", PLANS)
def test_dense_epilogue(dev, forced, plan, b_dtype):
    """The pages' NVFP4 x dense case carries the shared bias, gamma and
    scatter: all three, into a D with spare rows, on N = 256."""
    M, N, K = 300, 256, 1024
    bsg.bsg_force_plan(plan)
    p = workloads.make_dense(M, N, K, seed=3, b_dtype=b_dtype)
    e = workloads.make_epilogue(M, N, seed=8, m_out=M + 20, drop=0.2, bias_std=float(np.sqrt(K)))
    got = gpu_dense(p, dev, e["bias"], e["gamma"], e["scatter"], M + 20)
    _, T, ref = oracle_dense(p, bias=e["bias"], gamma=e["gamma"])
    dst = e["scatter"].numpy().astype(np.int64)
    live = dst >= 0
    assert_close(got[dst[live]], ref[live], T[live], f"{plan} epilogue")
    untouched = np.ones(M + 20, bool)
    untouched[dst[live]] = False
    assert (got[untouched] == SENTINEL).all()


def test_dense_worked_case(dev):
    """tests/golden/nvfp4_dense_case.txt exactly (K padded 32 -> 64 with zero
    codes, N 2 -> 8 with zero B rows)."""
    K, N = 64, 8
    codes = np.zeros((2, K), np.uint8)
    codes[0, :32] = 0x2
    codes[1, :32] = [k % 8 for k in range(32)]
    A = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))
    sfA = torch.tensor([[0x40, 0x30, 0x38, 0x38], [0x38, 0x38, 0x38, 0x38]], dtype=torch.uint8)
    B = torch.zeros((N, K), dtype=torch.bfloat16)
    B[0, :16], B[0, 16:32], B[1, :32] = 0.25, -3.0, 1.5
    p = dict(M=2, N=N, K=K, A=A, sfA=sfA, B=B, alpha=1.0)
    got = oracle.bf16_bits_to_float(gpu_dense(p, dev))
    assert got[:, :2].tolist() == [[-16.0, 60.0], [-99.0, 108.0]]


def test_dense_f16_worked_case(dev):
    """tests/golden/nvfp4_dense_f16_case.txt exactly (K padded 32 -> 64 with
    zero codes, N 2 -> 8 with zero B rows): a B value BF16 cannot hold, the
    smallest FP16 subnormal and the largest finite FP16 value."""
    K, N = 64, 8
    codes = np.zeros((1, K), np.uint8)
    codes[0, :16], codes[0, 16:32] = 0x2, 0x9
    A = torch.from_numpy((codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8))
    sfA = torch.tensor([[0x38, 0x48, 0x38, 0x38]], dtype=torch.uint8)
    Bb = np.zeros((N, K), np.uint16)
    Bb[0, :16], Bb[0, 16:32], Bb[1, :16], Bb[1, 16:32] = 0x3C01, 0x0001, 0x7BFF, 0xC000
    B = torch.from_numpy(Bb.view(np.int16)).view(torch.float16)
    p = dict(M=1, N=N, K=K, A=A, sfA=sfA, B=B, alpha=1.0)
    got = oracle.bf16_bits_to_float(gpu_dense(p, dev))
    assert got[0, :2].tolist() == [16.0, 1048576.0]


@pytest.mark.parametrize("b_dtype", DTYPES, ids=["bf16", "f16"])
def test_dense_4096_sampled(dev, b_dtype):
    """4096^3 in the default plan: sampled rows and columns of every tile."""
    M = N = K = 4096
    p = workloads.make_dense(M, N, K, seed=41, device=dev, b_dtype=b_dtype)
    got = gpu_dense(p, dev)
    rng = np.random.default_rng(4096)
    rows = sorted({int(t * 128 + rng.integers(128)) for t in range(M // 128)})
    cols = sorted({int(t * 256 + rng.integers(256)) for t in range(N // 256)})
    _, T, ref = oracle_dense(p, rows=rows)
    assert_close(got[rows], ref, T, "4096 rows")
    _, T, ref = oracle_dense(p, cols=cols[:8])
    assert_close(got[:, cols[:8]], ref, T, "4096 cols")
