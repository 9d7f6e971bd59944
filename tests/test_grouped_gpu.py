"""GPU parity of the grouped (ragged, routed) NVFP4 GEMM and its per-slice
scale layout against the CPU oracle.

"Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve Tensor-Memory
Failures", section "Ragged mode added routing rather than a plain matrix":
routed rows form slices, each multiplied by its own right-hand side. The
per-slice scale swizzle is compared bit for bit. The GEMM is compared
element by element under the GEMM tolerance on ragged splits: empty slices,
slices of a few rows, slices that end inside a warp's 32 rows or cross 128-row
tiles, ragged N, both 1-SM plans and the CTA pair's grouped mode (256-row
tile rows, a peer CTA whose rows lie past its slice loading no A), and the
epilogue variants (a bias per
slice, gamma, and the scatter back to token order). Rows of D that no row
names keep their prefill. The hand-worked case of
tests/golden/nvfp4_grouped_case.txt is checked exactly, and the MoE workload
(64 experts, 1024 tokens x top-8, 4096 x 7168) on sampled rows.
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
PLANS = [None, "nvfp4_tc1_128x128_s5_acc2", "nvfp4_tc1_128x256_s3_acc1", "nvfp4_tc2_256x256_s5_acc1"]


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


def gpu_swizzle_grouped(sf: torch.Tensor, offs: torch.Tensor, K: int, dev) -> np.ndarray:
    E, M = offs.numel() - 1, sf.shape[0]
    out = torch.full((bsg.nvfp4_grouped_scale_bytes(E, M, K),), 0xAB, dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales_grouped(E, M, K, offs.to(dev), sf.to(dev), out)
    torch.cuda.synchronize()
    return out.cpu().numpy()


def gpu_grouped(p, offs, dev, bias=None, gamma=None, scatter=None, m_out=None):
    E, M, N, K = p["E"], p["M"], p["N"], p["K"]
    m_out = M if m_out is None else m_out
    sa = torch.empty(bsg.nvfp4_grouped_scale_bytes(E, M, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales_grouped(E, M, K, offs.to(dev), p["sfA"].to(dev), sa)
    per = bsg.nvfp4_swizzled_scale_bytes(N, K)
    sb = torch.empty(E * per, dtype=torch.uint8, device=dev)
    for e in range(E):
        bsg.nvfp4_swizzle_scales(N, K, p["sfB"][e].to(dev).contiguous(), sb[e * per:(e + 1) * per])
    flat = torch.full((m_out * N + GUARD,), SENTINEL, dtype=torch.int16, device=dev)
    D = flat[: m_out * N].view(torch.bfloat16).view(m_out, N)
    dv = lambda t: None if t is None else t.to(dev)  # noqa: E731
    bsg.nvfp4_grouped_gemm(E, M, N, K, p["A"].to(dev), sa, p["B"].to(dev), sb, offs.to(dev), p["alpha"],
                           dv(bias), dv(gamma), dv(scatter), m_out, D)
    assert bsg.bsg_last_launch_count() == 1
    torch.cuda.synchronize()
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert (bits(flat[-GUARD:]) == SENTINEL).all(), "kernel wrote past the end of D"
    return bits(D)


def oracle_grouped(p, offs, bias=None, gamma=None):
    npy = lambda t: None if t is None else t.numpy()  # noqa: E731
    return oracle.get().nvfp4_grouped_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(), p["sfB"].numpy(),
                                           offs.numpy(), p["alpha"], p["K"], bias=npy(bias), gamma=npy(gamma))


def check(got, p, offs, bias, gamma, scatter, m_out, what):
    _, T, ref = oracle_grouped(p, offs, bias, gamma)
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


def offsets(sizes) -> torch.Tensor:
    o = np.zeros(len(sizes) + 1, np.int32)
    o[1:] = np.cumsum(sizes)
    return torch.from_numpy(o)


SPLITS = {
    "one_slice": [300],
    "ragged": [7, 0, 130, 1, 33, 129, 0, 64],
    "tiny": [1, 2, 3, 4, 5, 31, 32, 33],
    "empty_ends": [0, 0, 200, 56, 0],
    "many": [17 * (e % 5) for e in range(40)],
}


@pytest.mark.parametrize("split", list(SPLITS))
def test_grouped_scale_layout_bit_exact(dev, split):
    sizes = SPLITS[split]
    offs = offsets(sizes)
    M, K = int(offs[-1]), 1040 if split != "many" else 512
    if M == 0:
        pytest.skip("no rows")
    sf = torch.from_numpy(np.random.default_rng(M).integers(0, 256, (M, K // 16)).astype(np.uint8))
    want = oracle.get().swizzle_scales_grouped(sf.numpy(), offs.numpy(), K)
    assert np.array_equal(gpu_swizzle_grouped(sf, offs, K, dev), want)


def test_grouped_scale_layout_vector_path(dev):
    """K/16 a multiple of 16 (the 16-byte load path) over 4096 rows in 9 slices."""
    offs = offsets([500, 0, 1000, 127, 129, 1200, 1, 139, 1000])
    M, K = int(offs[-1]), 4096
    sf = torch.from_numpy(np.random.default_rng(9).integers(0, 256, (M, K // 16)).astype(np.uint8))
    assert np.array_equal(gpu_swizzle_grouped(sf, offs, K, dev),
                          oracle.get().swizzle_scales_grouped(sf.numpy(), offs.numpy(), K))


@pytest.mark.parametrize("split", list(SPLITS))
@pytest.mark.parametrize("plan", PLANS)
def test_grouped_gemm_splits(dev, forced, plan, split):
    sizes = SPLITS[split]
    offs = offsets(sizes)
    E, M, N, K = len(sizes), int(offs[-1]), 392, 1280
    bsg.bsg_force_plan(plan)
    p = workloads.make_grouped(E, M, N, K, seed=len(sizes) + M)
    got = gpu_grouped(p, offs, dev)
    check(got, p, offs, None, None, None, M, f"{plan} {split}")


@pytest.mark.parametrize("plan", PLANS)
def test_grouped_gemm_epilogue(dev, forced, plan):
    """A bias per slice, gamma per row, and the scatter back to token order
    of a top-3 routing of 100 tokens over 6 experts into a D with spare rows."""
    offs, dst = workloads.routing(6, 100, 3, seed=4)
    E, M, N, K = 6, 300, 520, 1024
    bsg.bsg_force_plan(plan)
    p = workloads.make_grouped(E, M, N, K, seed=6)
    rng = np.random.default_rng(2)
    bias = torch.from_numpy((rng.standard_normal((E, N)) * np.sqrt(K)).astype(np.float32))
    gamma = torch.from_numpy((1 + 0.5 * rng.standard_normal(M)).astype(np.float32))
    got = gpu_grouped(p, offs, dev, bias, gamma, dst, M + 11)
    check(got, p, offs, bias, gamma, dst, M + 11, f"{plan} epilogue")


def test_grouped_worked_case(dev):
    """tests/golden/nvfp4_grouped_case.txt, exactly: K padded from 16 to 256
    with zero codes, N from 2 to 8 with zero B rows and zero bias."""
    g = {}
    for line in (GOLDEN / "nvfp4_grouped_case.txt").read_text().splitlines():
        t = line.split()
        if t and not t[0].startswith("#"):
            g.setdefault(t[0], []).append(t[1:])
    K, N = 256, 8
    row = lambda c: [int(c, 16)] * 16 + [0] * (K - 16)  # noqa: E731
    pk = lambda c: (c[:, 0::2] | (c[:, 1::2] << 4)).contiguous()  # noqa: E731
    A = pk(torch.tensor([row(c) for c in g["acodes"][0]], dtype=torch.uint8))
    B = torch.stack([pk(torch.tensor([row(c) for c in g[f"b{e}codes"][0]] + [[0] * K] * (N - 2),
                                     dtype=torch.uint8)) for e in (0, 1)])
    M = A.shape[0]
    p = dict(E=2, M=M, N=N, K=K, A=A, B=B, sfA=torch.full((M, K // 16), 0x38, dtype=torch.uint8),
             sfB=torch.full((2, N, K // 16), 0x38, dtype=torch.uint8), alpha=float(g["alpha"][0][0]))
    offs = torch.tensor([int(v) for v in g["offs"][0]], dtype=torch.int32)
    got = oracle.bf16_bits_to_float(gpu_grouped(p, offs, dev))
    for r in g["plain"]:
        assert got[int(r[0]), :2].tolist() == [float(v) for v in r[1:]], ("plain", r[0], got[int(r[0])])
    bias = torch.zeros((2, N), dtype=torch.float32)
    bias[0, :2] = torch.tensor([float(v) for v in g["bias0"][0]])
    bias[1, :2] = torch.tensor([float(v) for v in g["bias1"][0]])
    gamma = torch.tensor([float(v) for v in g["gamma"][0]], dtype=torch.float32)
    got = oracle.bf16_bits_to_float(gpu_grouped(p, offs, dev, bias, gamma))
    for r in g["D"]:
        assert got[int(r[0]), :2].tolist() == [float(v) for v in r[1:]], ("D", r[0], got[int(r[0])])


@pytest.mark.parametrize("plan", ["nvfp4_tc1_128x128_s5_acc2", "nvfp4_tc1_128x256_s3_acc1", "nvfp4_tc2_256x256_s5_acc1"])
def test_single_slice_matches_plain_gemm(dev, forced, plan):
    """One slice over every row: the grouped kernel equals the plain kernel
    of the same plan bit for bit (zeros compared without sign)."""
    M, N, K = 520, 392, 2048
    bsg.bsg_force_plan(plan)
    p = workloads.make_grouped(1, M, N, K, seed=11)
    got = gpu_grouped(p, torch.tensor([0, M], dtype=torch.int32), dev)
    sa = torch.empty(bsg.nvfp4_swizzled_scale_bytes(M, K), dtype=torch.uint8, device=dev)
    sb = torch.empty(bsg.nvfp4_swizzled_scale_bytes(N, K), dtype=torch.uint8, device=dev)
    bsg.nvfp4_swizzle_scales(M, K, p["sfA"].to(dev), sa)
    bsg.nvfp4_swizzle_scales(N, K, p["sfB"][0].to(dev).contiguous(), sb)
    D = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    bsg.nvfp4_gemm_swizzled(M, N, K, p["A"].to(dev), sa, p["B"][0].to(dev).contiguous(), sb, p["alpha"], D)
    torch.cuda.synchronize()
    nz = lambda b: np.where((b & 0x7FFF) == 0, 0, b)  # noqa: E731
    assert np.array_equal(nz(got), nz(bits(D)))


def test_grouped_pair_most_slices(dev, forced):
    """The pair's slice table at its bound: 256 slices of 0 to 5 rows (about
    a third empty), ragged N, against the oracle."""
    sizes = [(7 * e) % 6 for e in range(256)]
    offs = offsets(sizes)
    E, M, N, K = 256, int(offs[-1]), 136, 512
    bsg.bsg_force_plan("nvfp4_tc2_256x256_s5_acc1")
    p = workloads.make_grouped(E, M, N, K, seed=256)
    got = gpu_grouped(p, offs, dev)
    check(got, p, offs, None, None, None, M, "pair, 256 slices")


def test_grouped_pair_slice_bound(dev, forced):
    """The pair's grouped mode takes at most 256 slices: forced beyond that,
    the call is refused before any launch."""
    E, N, K = 257, 136, 256
    offs = offsets([1] * E)
    p = workloads.make_grouped(E, E, N, K, seed=3)
    bsg.bsg_force_plan("nvfp4_tc2_256x256_s5_acc1")
    with pytest.raises(bsg.BsgError) as e:
        gpu_grouped(p, offs, dev)
    assert e.value.code == bsg.BSG_ERR_NO_PLAN


@pytest.mark.parametrize("plan", [None, "nvfp4_tc2_256x256_s5_acc1"])
def test_moe_workload_sampled(dev, forced, plan):
    """64 experts, 1024 tokens x top-8 (8192 routed rows), 4096 x 7168, in the
    launch configuration the benchmark times, with the scatter back to token
    order: sampled rows of every slice against the oracle."""
    bsg.bsg_force_plan(plan)
    w = workloads.GROUPED_WORKLOADS["moe_e64_t1024_k8"]
    offs, dst = workloads.routing(w.E, w.tokens, w.top_k, seed=1)
    p = workloads.make_grouped(w.E, w.M, w.N, w.K, seed=1, device=dev)     # 0.94 GB of weights
    got = gpu_grouped(p, offs, dev, scatter=dst, m_out=w.M)
    A, sfA = p["A"].cpu().numpy(), p["sfA"].cpu().numpy()
    o = offs.numpy()
    rng = np.random.default_rng(64)
    rows = sorted({int(o[e] + rng.integers(o[e + 1] - o[e])) for e in range(w.E) if o[e + 1] > o[e]}
                  | {0, w.M - 1})
    ref_rows = []
    sub = {}
    for e in range(w.E):
        rs = [r for r in rows if o[e] <= r < o[e + 1]]
        if not rs:
            continue
        _, T, ref = oracle.get().nvfp4_gemm(A[o[e]:o[e + 1]], sfA[o[e]:o[e + 1]], p["B"][e].cpu().numpy(),
                                            p["sfB"][e].cpu().numpy(), p["alpha"], w.K,
                                            rows=[r - int(o[e]) for r in rs])
        for i, r in enumerate(rs):
            sub[r] = (T[i], ref[i])
        ref_rows += rs
    d = dst.numpy().astype(np.int64)
    for r in ref_rows:
        T, ref = sub[r]
        assert oracle.within_tolerance(got[d[r]][None], ref[None], T[None]).all(), f"row {r}"
