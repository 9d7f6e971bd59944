"""Seeded synthetic inputs for the block-scaled GEMM.

Shared by the tests, the smoke check and the benchmark. This module only
draws random numbers and encodes them into the operand formats (E2M1 codes
packed two per byte, E4M3 scale bytes, E4M3 FP8 operands). It holds none of
the GEMM's arithmetic, imports neither the oracle nor the library, and both
sides receive exactly the bytes it produces.

Workloads (the pages' shapes; all data synthetic):
  * ``nvfp4_256``   M=N=K=256, E2M1 codes uniform over all 16 nibbles, block
    scales 2^u with u uniform in [-4, 4], alpha = 1.
  * ``nvfp4_4096``  M=N=K=4096, N(0,1) rounded to BF16, two-level NVFP4
    quantisation (below), alpha = 1 / (s_gA * s_gB).
  * ``nvfp4_16384`` M=N=K=16384, as ``nvfp4_4096`` (the square shape of the
    ring-depth sweep in "Together AI Ports ThunderKittens GEMM Kernels to
    NVIDIA Vera Rubin NVL72", "Building the GEMM").
  * ``fp8_8192``    M=N=K=8192 E4M3 from N(0,1) with per-tensor scale
    amax/448, alpha = s_A * s_B.
  * skinny cells   M in {64,128,256,512} x (N,K) in {(3072,3072),
    (12288,3072), (3072,12288)}, activations and weights N(0, 0.02), two-level
    NVFP4.

Two-level NVFP4 quantisation of a tensor x (input generation only):
  s_g = 448*6 / amax|x| (FP32); per 16-block b: scale_b = E4M3_rne(min(448,
  amax_b/6 * s_g)); code = E2M1_rne_sat(x * s_g / scale_b) (code 0 where
  scale_b = 0). The GEMM then needs alpha = 1/(s_gA * s_gB).

Random numbers come from ``torch.Generator`` on the device the data is made
on, so CPU and GPU draws differ in bits but not in distribution; every parity
check feeds the same bytes to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

SEED_BASE = 0xB5C0


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str          # "nvfp4" or "fp8"
    M: int
    N: int
    K: int
    dist: str          # "uniform_codes" or "normal"
    std: float = 1.0
    index: int = 0     # seed slot

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> float:
        """Minimum HBM bytes of one GEMM: packed operands, scales, BF16 D."""
        if self.kind == "nvfp4":
            return (self.M + self.N) * self.K * 9 / 16 + 2.0 * self.M * self.N
        return (self.M + self.N) * self.K + 2.0 * self.M * self.N


SKINNY_M = (64, 128, 256, 512)
SKINNY_NK = ((3072, 3072), (12288, 3072), (3072, 12288))

WORKLOADS: dict[str, Workload] = {}


def _add(w: Workload) -> None:
    WORKLOADS[w.name] = w


_add(Workload("nvfp4_256", "nvfp4", 256, 256, 256, "uniform_codes", index=0))
_add(Workload("nvfp4_4096", "nvfp4", 4096, 4096, 4096, "normal", 1.0, index=1))
_add(Workload("nvfp4_16384", "nvfp4", 16384, 16384, 16384, "normal", 1.0, index=2))
_add(Workload("fp8_8192", "fp8", 8192, 8192, 8192, "normal", 1.0, index=3))
for _n, _k in SKINNY_NK:
    for _m in SKINNY_M:
        _add(Workload(f"nvfp4_skinny_m{_m}_n{_n}_k{_k}", "nvfp4", _m, _n, _k, "normal", 0.02,
                      index=4))


def seed_for(w: Workload, operand: int) -> int:
    """operand 0 = A (activations), 1 = B (weights)."""
    return SEED_BASE + 16 * w.index + operand + 1000 * (w.M + 7 * w.N + 13 * w.K)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


# --------------------------------------------------------------------------
# Encoders (inputs only)
# --------------------------------------------------------------------------

def e2m1_encode(v: torch.Tensor) -> torch.Tensor:
    """Nearest E2M1 code (ties to even mantissa, saturating at 6), uint8 0..15."""
    mag = v.abs()
    idx = ((mag > 0.25).to(torch.uint8) + (mag >= 0.75).to(torch.uint8)
           + (mag > 1.25).to(torch.uint8) + (mag >= 1.75).to(torch.uint8)
           + (mag > 2.5).to(torch.uint8) + (mag >= 3.5).to(torch.uint8)
           + (mag > 5.0).to(torch.uint8))
    return idx | ((v < 0).to(torch.uint8) << 3)


def pack_e2m1(codes: torch.Tensor) -> torch.Tensor:
    """uint8 codes [rows, K] -> bytes [rows, K/2]; element 2i in the low nibble."""
    lo = codes[:, 0::2]
    hi = codes[:, 1::2]
    return (lo | (hi << 4)).contiguous()


def unpack_e2m1(packed: torch.Tensor) -> torch.Tensor:
    """bytes [rows, K/2] -> uint8 codes [rows, K] (inverse of ``pack_e2m1``)."""
    rows, half = packed.shape
    out = torch.empty((rows, 2 * half), dtype=torch.uint8, device=packed.device)
    out[:, 0::2] = packed & 15
    out[:, 1::2] = packed >> 4
    return out


def e4m3_encode(v: torch.Tensor) -> torch.Tensor:
    """Nearest E4M3 code (ties to even) of values clamped to [-448, 448]."""
    return v.clamp(-448.0, 448.0).to(torch.float8_e4m3fn).view(torch.uint8)


def nvfp4_quantise(x: torch.Tensor):
    """Two-level NVFP4 encoding of float32 x[rows, K] -> (packed, sf, s_g)."""
    rows, K = x.shape
    amax = x.abs().amax().float()
    s_g = torch.where(amax > 0, (448.0 * 6.0) / amax, torch.ones_like(amax)).float()
    xb = x.reshape(rows, K // 16, 16)
    bmax = xb.abs().amax(-1)
    sf = e4m3_encode((bmax / 6.0 * s_g).clamp(max=448.0))
    sf_val = sf.view(torch.float8_e4m3fn).to(torch.float32)
    safe = torch.where(sf_val > 0, sf_val, torch.ones_like(sf_val))
    scaled = xb * s_g / safe.unsqueeze(-1)
    codes = e2m1_encode(scaled)
    codes = torch.where((sf_val > 0).unsqueeze(-1), codes, torch.zeros_like(codes))
    return pack_e2m1(codes.reshape(rows, K)), sf.contiguous(), float(s_g)


def normal_bf16(rows: int, K: int, seed: int, std: float, device) -> torch.Tensor:
    """N(0, std^2) float32, rounded through BF16 as the source activations."""
    x = torch.randn((rows, K), generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(torch.bfloat16).to(torch.float32)


def uniform_nvfp4(rows: int, K: int, seed: int, device):
    """All 16 E2M1 codes uniformly; block scales 2^u, u uniform in [-4, 4]."""
    g = _gen(seed, device)
    packed = torch.randint(0, 256, (rows, K // 2), generator=g, device=device,
                           dtype=torch.int32).to(torch.uint8)
    u = torch.randint(-4, 5, (rows, K // 16), generator=g, device=device, dtype=torch.int32)
    sf = ((u + 7) << 3).to(torch.uint8)   # E4M3 code of 2^u: exponent field u+7
    return packed, sf


# --------------------------------------------------------------------------
# Whole problems
# --------------------------------------------------------------------------

def make_nvfp4(w: Workload, device="cpu", M: int | None = None, N: int | None = None,
               K: int | None = None) -> dict:
    """A, sfA, B, sfB (uint8 tensors on ``device``) and alpha for workload w.

    M, N, K override the workload's sizes (same recipe, e.g. for ragged tests).
    """
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    if w.dist == "uniform_codes":
        A, sfA = uniform_nvfp4(M, K, seed_for(w, 0), device)
        B, sfB = uniform_nvfp4(N, K, seed_for(w, 1), device)
        alpha = 1.0
    else:
        A, sfA, sga = nvfp4_quantise(normal_bf16(M, K, seed_for(w, 0), w.std, device))
        B, sfB, sgb = nvfp4_quantise(normal_bf16(N, K, seed_for(w, 1), w.std, device))
        alpha = float(torch.tensor(1.0, dtype=torch.float32)
                      / (torch.tensor(sga, dtype=torch.float32) * torch.tensor(sgb, dtype=torch.float32)))
    return dict(M=M, N=N, K=K, A=A, sfA=sfA, B=B, sfB=sfB, alpha=alpha)


def make_fp8(w: Workload, device="cpu", M: int | None = None, N: int | None = None,
             K: int | None = None) -> dict:
    """E4M3 A, B (uint8) with alpha = s_A * s_B, s = amax/448 per tensor."""
    M = w.M if M is None else M
    N = w.N if N is None else N
    K = w.K if K is None else K
    out = dict(M=M, N=N, K=K)
    scales = []
    for name, rows, op in (("A", M, 0), ("B", N, 1)):
        x = normal_bf16(rows, K, seed_for(w, op), w.std, device)
        amax = x.abs().amax().float()
        s = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax)).float()
        out[name] = e4m3_encode(x / s).contiguous()
        scales.append(s)
    out["alpha"] = float((scales[0] * scales[1]).float())
    return out


def make_epilogue(M: int, N: int, seed: int, m_out: int | None = None, drop: float = 0.0,
                  bias_std: float = 1.0, device="cpu") -> dict:
    """Inputs of the GEMM epilogue variants ("Triton #11171 - Why Two New
    NVFP4 Test Cases Produced Twelve Tensor-Memory Failures", the scatter,
    gamma and shared-bias sections; the pages give no distributions):

      bias    float32[N] ~ N(0, bias_std^2)
      gamma   float32[M] ~ N(1, 0.5^2)  (mostly positive, some negative)
      scatter int32[M]: a random injective map of the computed rows into
              [0, m_out) (m_out >= M, default M: a random permutation), a
              fraction ``drop`` of its entries then set to -1 (not written)
    """
    m_out = M if m_out is None else m_out
    if m_out < M:
        raise ValueError("an injective scatter needs m_out >= M")
    g = _gen(SEED_BASE + 7919 * seed + 31 * M + N, "cpu")
    bias = (torch.randn(N, generator=g, dtype=torch.float32) * bias_std).contiguous()
    gamma = (1.0 + 0.5 * torch.randn(M, generator=g, dtype=torch.float32)).contiguous()
    scatter = torch.randperm(m_out, generator=g)[:M].to(torch.int32)
    if drop > 0:
        scatter[torch.rand(M, generator=g) < drop] = -1
    return {k: v.to(device) for k, v in dict(bias=bias, gamma=gamma, scatter=scatter).items()}


# --------------------------------------------------------------------------
# Grouped (ragged, routed) GEMM inputs
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class GroupedWorkload:
    """An MoE expert matmul: `tokens` tokens each routed to `top_k` distinct
    experts out of `E` (uniformly, seeded), so M = tokens * top_k routed rows
    in slices of ragged size; every expert's weights are N x K."""
    name: str
    E: int
    tokens: int
    top_k: int
    N: int
    K: int
    index: int = 5

    @property
    def M(self) -> int:
        return self.tokens * self.top_k

    @property
    def flops(self) -> float:
        return 2.0 * self.M * self.N * self.K

    @property
    def algorithmic_bytes(self) -> float:
        """Packed A and all E weight matrices with their scales, BF16 D."""
        return (self.M + self.E * self.N) * self.K * 9 / 16 + 2.0 * self.M * self.N


GROUPED_WORKLOADS: dict[str, GroupedWorkload] = {
    # 1024 tokens x top-8 of 64 experts (about 128 rows per expert), expert
    # up-projection 4096 x 7168
    "moe_e64_t1024_k8": GroupedWorkload("moe_e64_t1024_k8", 64, 1024, 8, 4096, 7168),
}


def routing(E: int, tokens: int, top_k: int, seed: int):
    """Route each token to top_k distinct experts (uniform, seeded); the
    routed rows sorted by (expert, token). Returns (offs int32[E+1], dst
    int32[M]) where dst[row] = token * top_k + slot: the row's place in
    token order (the scatter back from expert order)."""
    g = _gen(SEED_BASE + 104729 * seed + E, "cpu")
    choice = torch.stack([torch.randperm(E, generator=g)[:top_k] for _ in range(tokens)])   # [tokens, top_k]
    expert = choice.reshape(-1)                        # row t*top_k + s -> expert
    order = torch.sort(expert * tokens + torch.arange(tokens).repeat_interleave(top_k), stable=True).indices
    counts = torch.bincount(expert, minlength=E)
    offs = torch.zeros(E + 1, dtype=torch.int32)
    offs[1:] = torch.cumsum(counts, 0).to(torch.int32)
    return offs, order.to(torch.int32)


def make_grouped(E: int, M: int, N: int, K: int, seed: int, device="cpu", std: float = 1.0) -> dict:
    """A [M][K/2] + row-major sfA, B [E][N][K/2] + sfB [E][N][K/16] (one
    two-level quantisation over all E * N weight rows, so one alpha serves
    every slice), from N(0, std^2) through BF16."""
    A, sfA, sga = nvfp4_quantise(normal_bf16(M, K, SEED_BASE + 7 * seed, std, device))
    B, sfB, sgb = nvfp4_quantise(normal_bf16(E * N, K, SEED_BASE + 7 * seed + 1, std, device))
    alpha = float(torch.tensor(1.0, dtype=torch.float32)
                  / (torch.tensor(sga, dtype=torch.float32) * torch.tensor(sgb, dtype=torch.float32)))
    return dict(E=E, M=M, N=N, K=K, A=A, sfA=sfA, B=B.reshape(E, N, K // 2), sfB=sfB.reshape(E, N, K // 16),
                alpha=alpha)


def make_dense_grouped(E: int, M: int, N: int, K: int, seed: int, device="cpu", std: float = 1.0,
                       b_dtype: torch.dtype = torch.bfloat16) -> dict:
    """Grouped NVFP4 x dense inputs: A two-level NVFP4 (row-major sfA) from
    N(0, std^2) through BF16, B [E][N][K] = N(0, std^2) drawn in FP32 and
    rounded to b_dtype, alpha = 1 / s_gA."""
    A, sfA, sga = nvfp4_quantise(normal_bf16(M, K, SEED_BASE + 13 * seed, std, device))
    B = torch.randn((E * N, K), generator=_gen(SEED_BASE + 13 * seed + 1, device), device=device,
                    dtype=torch.float32)
    B = (B * std if std != 1.0 else B).to(b_dtype).reshape(E, N, K).contiguous()
    alpha = float(torch.tensor(1.0, dtype=torch.float32) / torch.tensor(sga, dtype=torch.float32))
    return dict(E=E, M=M, N=N, K=K, A=A, sfA=sfA, B=B, alpha=alpha)


def make_dense(M: int, N: int, K: int, seed: int, device="cpu", std: float = 1.0,
               b_dtype: torch.dtype = torch.bfloat16) -> dict:
    """NVFP4 x dense inputs: A two-level NVFP4 (row-major sfA) from
    N(0, std^2) through BF16, B = N(0, std^2) drawn in FP32 and rounded to
    b_dtype (torch bfloat16 or float16, [N][K]), alpha = 1 / s_gA."""
    A, sfA, sga = nvfp4_quantise(normal_bf16(M, K, SEED_BASE + 11 * seed, std, device))
    B = torch.randn((N, K), generator=_gen(SEED_BASE + 11 * seed + 1, device), device=device, dtype=torch.float32)
    B = (B * std if std != 1.0 else B).to(b_dtype).contiguous()
    alpha = float(torch.tensor(1.0, dtype=torch.float32) / torch.tensor(sga, dtype=torch.float32))
    return dict(M=M, N=N, K=K, A=A, sfA=sfA, B=B, alpha=alpha)
