"""Pins of the CPU oracle against facts fixed outside the oracle itself.

Every pin below checks the oracle against something it does not compute:
golden tables from the format specifications (``tests/golden/``), values
worked by hand, a library decoder (PyTorch's CPU float8_e4m3fn), exact
rational arithmetic, an independent numpy restatement, and invariants of the
definition. ``test_planted_mistake_is_caught`` compiles the oracle with one
deliberate mistake at a time (a wrong exponent bias, a dropped sign, swapped
nibbles in one operand, a dropped scale, a dropped block, a transposed operand, a wrong
scale layout; in the quantiser, ties rounded away from zero, a dropped global
scale, swapped nibbles, block scales rounded up; in the epilogue, gamma
applied before the bias, bias indexed by row; in the grouped GEMM, a slice
multiplied by the next slice's right-hand side; in the NVFP4 x dense GEMM,
A's block scales dropped; in Freivalds' full-product check, B's block scales
dropped, the random vector read backwards, magnitudes summed with their
signs) and shows that at least one pin fails for each.
"""
from __future__ import annotations

import math
import random
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
import workloads

GOLDEN = Path(__file__).resolve().parent / "golden"


# --------------------------------------------------------------------------
# Golden data
# --------------------------------------------------------------------------

def _rows(name):
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.strip()
        if line and not line.startswith("#"):
            yield line.split()


E2M1_TABLE = {int(c, 16): float(v) for c, v in _rows("e2m1_table.txt")}
E4M3_POINTS = {int(c, 16): float(v) for c, v in _rows("e4m3_points.txt")}
BF16_CASES = [(float.fromhex(x), int(b, 16)) for x, b, *_ in _rows("bf16_rne_cases.txt")]


def e4m3_lib(code: int) -> float:
    """PyTorch's own E4M3 decoder (a library routine, used only as a check)."""
    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn)
                 .to(torch.float64)[0])


def e4m3_code_of(value: float) -> int:
    """E4M3 code of an exactly representable value, via PyTorch's encoder."""
    return int(torch.tensor([value], dtype=torch.float32).to(torch.float8_e4m3fn)
               .view(torch.uint8)[0])


def pack(codes: np.ndarray) -> np.ndarray:
    """uint8 codes [rows, K] -> packed bytes, element 2i in the low nibble."""
    codes = np.asarray(codes, np.uint8)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)


def deq_nvfp4(packed: np.ndarray, sf: np.ndarray) -> np.ndarray:
    """Independent dequantisation via the golden E2M1 table and torch E4M3."""
    lo = packed & 15
    hi = packed >> 4
    codes = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    codes[:, 0::2] = lo
    codes[:, 1::2] = hi
    tab = np.array([E2M1_TABLE[c] for c in range(16)])
    scale = np.array([e4m3_lib(c) for c in range(256)])
    return tab[codes] * np.repeat(scale[sf], 16, axis=1)


# --------------------------------------------------------------------------
# Pins: each takes an Oracle and raises AssertionError on a mismatch
# --------------------------------------------------------------------------

def pin_e2m1_table(o):
    for code, val in E2M1_TABLE.items():
        got = o.e2m1(code)
        assert got == val and math.copysign(1, got) == math.copysign(1, val), (code, got, val)


def pin_e4m3_codes(o):
    for code in range(256):
        got, ref = o.e4m3(code), e4m3_lib(code)
        assert (math.isnan(got) and math.isnan(ref)) or got == ref, (code, got, ref)
    for code, val in E4M3_POINTS.items():
        got = o.e4m3(code)
        assert (math.isnan(got) and math.isnan(val)) or got == val, (code, got, val)


def pin_bf16_cases(o):
    for x, bits in BF16_CASES:
        assert o.bf16_rne(x) == bits, (x.hex(), hex(o.bf16_rne(x)), hex(bits))
    # binary32-representable inputs: PyTorch's float32 -> bfloat16 (RNE) is
    # then a single rounding too, so the two must agree bit for bit.
    rng = np.random.default_rng(7)
    f = np.concatenate([
        rng.standard_normal(3000).astype(np.float32) * np.float32(1e3),
        (rng.integers(-2**15, 2**15, 2000).astype(np.float32) * np.float32(2.0 ** -8)),
        np.array([1e-39, -3e-40, 1e-45, 3.4e38, -3.39e38], np.float32),
    ])
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().astype(np.uint16)
    for x, r in zip(f.tolist(), ref.tolist()):
        assert o.bf16_rne(x) == r, (x, hex(o.bf16_rne(x)), hex(r))


def pin_worked_1x1x16(o):
    # A[0][t] = B[0][t] = code t (t = 0..15): values 0, .5, 1, 1.5, 2, 3, 4, 6
    # and their negatives. sfA = 2.0 (0x40), sfB = 0.5 (0x30), alpha = 1.
    # sum_t a_t^2 = 2 * (0 + .25 + 1 + 2.25 + 4 + 9 + 16 + 36) = 137, so
    # D = 2 * 0.5 * 137 = 137, exact in BF16 (0x4309).
    codes = np.arange(16, dtype=np.uint8)[None, :]
    A = pack(codes)
    S, T, D = o.nvfp4_gemm(A, np.array([[0x40]], np.uint8), A, np.array([[0x30]], np.uint8), 1.0, 16)
    assert S[0, 0] == 137.0 and T[0, 0] == 137.0 and D[0, 0] == 0x4309, (S, T, D)


def pin_worked_2x2x32(o):
    # A0 = all 1.0, sA0 = [1, 2];  A1 = all -1.0, sA1 = [0.5, 1]
    # B0 = all 2.0, sB0 = [1, 1];  B1 = code (k mod 8) (each 16-block sums to
    # 36), sB1 = [1, 0.25].
    # D00 = 32 + 64 = 96; D01 = 36 + 18 = 54; D10 = -16 - 32 = -48;
    # D11 = -18 - 9 = -27.
    A = pack(np.array([[0x2] * 32, [0xA] * 32], np.uint8))
    B = pack(np.array([[0x4] * 32, [k % 8 for k in range(32)]], np.uint8))
    sfA = np.array([[0x38, 0x40], [0x30, 0x38]], np.uint8)
    sfB = np.array([[0x38, 0x38], [0x38, 0x28]], np.uint8)
    S, _, D = o.nvfp4_gemm(A, sfA, B, sfB, 1.0, 32)
    assert np.array_equal(S, [[96.0, 54.0], [-48.0, -27.0]]), S
    assert np.array_equal(oracle.bf16_bits_to_float(D), S), D


def pin_one_hot(o):
    # A row i is one-hot at k = pi(i) with value 1.0, all scales 1.0, alpha 1:
    # then D[i][j] is exactly the E2M1 value of B[j][pi(i)]. Positions of both
    # parities pin that A and B are read with the same nibble order (element
    # 2i in the low nibble, as packed here).
    K, M, N = 64, 64, 48
    rng = np.random.default_rng(11)
    pi = rng.permutation(K)[:M]
    codes_a = np.zeros((M, K), np.uint8)
    codes_a[np.arange(M), pi] = 0x2
    codes_b = rng.integers(0, 16, (N, K)).astype(np.uint8)
    ones_a = np.full((M, K // 16), 0x38, np.uint8)
    ones_b = np.full((N, K // 16), 0x38, np.uint8)
    S, _, _ = o.nvfp4_gemm(pack(codes_a), ones_a, pack(codes_b), ones_b, 1.0, K)
    tab = np.array([E2M1_TABLE[c] for c in range(16)])
    want = tab[codes_b[:, pi]].T
    assert np.array_equal(S, want)


def pin_brute_force_k16(o):
    # K = 16, a single nonzero position t: row i of A holds code i at t, row j
    # of B holds code j at t; per-row scales vary. Then S[i][j] is the table
    # product e2m1(i) * e2m1(j) * sA_i * sB_j for all 16 x 16 code pairs.
    tab = np.array([E2M1_TABLE[c] for c in range(16)])
    scale_codes = [0x38, 0x40, 0x30, 0x3C, 0x01, 0x7E, 0x55, 0x23]
    for t in range(16):
        ca = np.zeros((16, 16), np.uint8)
        ca[:, t] = np.arange(16)
        sa = np.array([[scale_codes[(i + t) % 8]] for i in range(16)], np.uint8)
        sb = np.array([[scale_codes[(3 * j + t) % 8]] for j in range(16)], np.uint8)
        S, T, _ = o.nvfp4_gemm(pack(ca), sa, pack(ca), sb, 1.0, 16)
        vs_a = np.array([e4m3_lib(int(c)) for c in sa[:, 0]])
        vs_b = np.array([e4m3_lib(int(c)) for c in sb[:, 0]])
        want = np.outer(tab * vs_a, tab * vs_b)
        assert np.array_equal(S, want), t
        assert np.array_equal(T, np.abs(want)), t


def _uniform_problem(M, N, K, seed):
    w = workloads.WORKLOADS["nvfp4_256"]
    g = torch.Generator().manual_seed(seed)
    A = torch.randint(0, 256, (M, K // 2), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    B = torch.randint(0, 256, (N, K // 2), generator=g, dtype=torch.int32).to(torch.uint8).numpy()
    sfA = workloads.uniform_nvfp4(M, K, seed + 1, "cpu")[1].numpy()
    sfB = workloads.uniform_nvfp4(N, K, seed + 2, "cpu")[1].numpy()
    del w
    return A, sfA, B, sfB


def pin_scale_linearity(o):
    # Doubling one block scale sfA[i][b] (E4M3 exponent field + 1) adds
    # exactly that block's contribution to row i and leaves other rows alone.
    M = N = 32
    K = 64
    A, sfA, B, sfB = _uniform_problem(M, N, K, 3)
    S0, _, _ = o.nvfp4_gemm(A, sfA, B, sfB, 1.0, K)
    i, b = 5, 2
    sf2 = sfA.copy()
    assert ((sf2[i, b] >> 3) & 15) < 14
    sf2[i, b] += 8
    S1, _, _ = o.nvfp4_gemm(A, sf2, B, sfB, 1.0, K)
    blk, _, _ = o.nvfp4_gemm(A[:, 8 * b:8 * b + 8], sfA[:, b:b + 1], B[:, 8 * b:8 * b + 8],
                             sfB[:, b:b + 1], 1.0, 16)
    assert np.array_equal(S1[i] - S0[i], blk[i])
    others = np.arange(M) != i
    assert np.array_equal(S1[others], S0[others])
    # halving a scale (exponent field - 1) removes half the contribution
    sf3 = sfA.copy()
    sf3[i, b] -= 8
    S3, _, _ = o.nvfp4_gemm(A, sf3, B, sfB, 1.0, K)
    assert np.array_equal(S0[i] - S3[i], blk[i] / 2)


def pin_numpy_definition(o):
    # Independent restatement: dequantise with the golden E2M1 table and the
    # library E4M3 decoder, multiply with numpy in float64. With 2^u scales
    # every partial sum is exact in double, so the results must be identical.
    # Square so that a transposed operand cannot hide.
    M = N = K = 64
    A, sfA, B, sfB = _uniform_problem(M, N, K, 9)
    S, T, D = o.nvfp4_gemm(A, sfA, B, sfB, 0.75, K)
    da, db = deq_nvfp4(A, sfA), deq_nvfp4(B, sfB)
    assert np.array_equal(S, 0.75 * (da @ db.T))
    assert np.array_equal(T, 0.75 * (np.abs(da) @ np.abs(db).T))
    # and through a rectangular, N(0,1)-quantised problem (not exact sums)
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=48, N=80, K=256)
    S, _, _ = o.nvfp4_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(), p["sfB"].numpy(),
                           p["alpha"], 256)
    ref = float(np.float32(p["alpha"])) * (deq_nvfp4(p["A"].numpy(), p["sfA"].numpy())
                                           @ deq_nvfp4(p["B"].numpy(), p["sfB"].numpy()).T)
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())


def pin_fraction_exact(o):
    # Brute force in exact rational arithmetic on a tiny problem.
    M, N, K = 3, 5, 32
    rng = random.Random(5)
    ca = [[rng.randrange(16) for _ in range(K)] for _ in range(M)]
    cb = [[rng.randrange(16) for _ in range(K)] for _ in range(N)]
    sa = [[rng.choice([0x38, 0x41, 0x2A, 0x06, 0x7E]) for _ in range(K // 16)] for _ in range(M)]
    sb = [[rng.choice([0x38, 0x3B, 0x49, 0x11]) for _ in range(K // 16)] for _ in range(N)]
    alpha = 0.3125
    S, _, D = o.nvfp4_gemm(pack(np.array(ca, np.uint8)), np.array(sa, np.uint8),
                           pack(np.array(cb, np.uint8)), np.array(sb, np.uint8), alpha, K)
    for i in range(M):
        for j in range(N):
            acc = Fraction(0)
            for k in range(K):
                acc += (Fraction(E2M1_TABLE[ca[i][k]]) * Fraction(E2M1_TABLE[cb[j][k]])
                        * Fraction(e4m3_lib(sa[i][k // 16])) * Fraction(e4m3_lib(sb[j][k // 16])))
            exact = Fraction(alpha) * acc
            assert Fraction(S[i, j]) == exact, (i, j)
            # BF16 of the exact value: nearest of the two neighbours, by hand
            assert D[i, j] == o.bf16_rne(float(exact))


def pin_fp8_numpy(o):
    # FP8: library-decoded E4M3 operands multiplied by numpy in float64; all
    # partial sums are exact in double at this size, so only the final scale
    # multiplication can round.
    w = workloads.WORKLOADS["fp8_8192"]
    p = workloads.make_fp8(w, "cpu", M=40, N=24, K=96)
    A, B = p["A"].numpy(), p["B"].numpy()
    S, T, _ = o.fp8_gemm(A, B, p["alpha"], 1.0, 1.0)
    dec = np.array([e4m3_lib(c) for c in range(256)])
    ref = (dec[A] @ dec[B].T) * float(np.float32(p["alpha"]))
    assert np.allclose(S, ref, rtol=1e-15, atol=0)
    # per-tensor scales: alpha*sA*sB with the three FP32 values
    S2, _, _ = o.fp8_gemm(A, B, 2.0, 0.5, 3.0)
    assert np.allclose(S2, (dec[A] @ dec[B].T) * 3.0, rtol=1e-15, atol=0)
    assert np.array_equal(T, (np.abs(dec[A]) @ np.abs(dec[B]).T) * float(np.float32(p["alpha"])))


def pin_epilogue_worked(o):
    """Bias, gamma and scatter on the hand-worked case of
    tests/golden/nvfp4_epilogue_case.txt (values and signs exact)."""
    g = {}
    for t in _rows("nvfp4_epilogue_case.txt"):
        g.setdefault(t[0], []).append(t[1:])
    ac = [int(c, 16) for c in g["acodes"][0]]
    bc = [int(c, 16) for c in g["bcodes"][0]]
    A = pack(np.array([[c] * 16 for c in ac], np.uint8))
    B = pack(np.array([[c] * 16 for c in bc], np.uint8))
    sfA = np.full((len(ac), 1), 0x38, np.uint8)
    sfB = np.full((len(bc), 1), 0x38, np.uint8)
    bias = np.array([float(v) for v in g["bias"][0]], np.float32)
    gamma = np.array([float(v) for v in g["gamma"][0]], np.float32)
    S, T, D = o.nvfp4_gemm(A, sfA, B, sfB, float(g["alpha"][0][0]), 16, bias=bias, gamma=gamma)
    Dv = oracle.bf16_bits_to_float(D)
    for r in g["D"]:
        i = int(r[0])
        want = [float(v) for v in r[1:]]
        assert S[i].tolist() == want and Dv[i].tolist() == want, (i, S[i], want)
        assert [math.copysign(1, v) for v in Dv[i]] == [math.copysign(1, v) for v in want], i
    for r in g["T"]:
        assert T[int(r[0])].tolist() == [float(v) for v in r[1:]], ("T", r[0])
    out = np.full(D.shape, 0x7FC0, np.uint16)
    o.scatter_rows(D, [int(v) for v in g["scatter"][0]], out)
    outv = oracle.bf16_bits_to_float(out)
    for r in g["out"]:
        want = np.array([float(v) for v in r[1:]])
        got = outv[int(r[0])]
        assert np.array_equal(np.isnan(got), np.isnan(want)), r[0]
        assert np.array_equal(got[~np.isnan(want)], want[~np.isnan(want)]), (r[0], got, want)


def pin_epilogue_numpy(o):
    # Independent restatement of the epilogue in numpy (float64) on a
    # rectangular problem with 2^u scales (all sums exact): bias broadcast
    # over rows, gamma over columns, bias before gamma. Also FP8.
    M, N, K = 24, 40, 64
    A, sfA, B, sfB = _uniform_problem(M, N, K, 13)
    rng = np.random.default_rng(4)
    bias = rng.standard_normal(N).astype(np.float32)
    gamma = rng.standard_normal(M).astype(np.float32)
    S, T, _ = o.nvfp4_gemm(A, sfA, B, sfB, 0.75, K, bias=bias, gamma=gamma)
    da, db = deq_nvfp4(A, sfA), deq_nvfp4(B, sfB)
    ref = (0.75 * (da @ db.T) + bias.astype(np.float64)[None, :]) * gamma.astype(np.float64)[:, None]
    assert np.allclose(S, ref, rtol=1e-15, atol=0)
    Tref = (0.75 * (np.abs(da) @ np.abs(db).T) + np.abs(bias.astype(np.float64))[None, :]) \
        * np.abs(gamma.astype(np.float64))[:, None]
    assert np.allclose(T, Tref, rtol=1e-15, atol=0)
    # gamma alone and bias alone
    Sg, _, _ = o.nvfp4_gemm(A, sfA, B, sfB, 0.75, K, gamma=gamma)
    assert np.allclose(Sg, 0.75 * (da @ db.T) * gamma.astype(np.float64)[:, None], rtol=1e-15, atol=0)
    Sb, _, _ = o.nvfp4_gemm(A, sfA, B, sfB, 0.75, K, bias=bias)
    assert np.allclose(Sb, 0.75 * (da @ db.T) + bias.astype(np.float64)[None, :], rtol=1e-15, atol=0)
    w = workloads.WORKLOADS["fp8_8192"]
    p = workloads.make_fp8(w, "cpu", M=M, N=N, K=96)
    dec = np.array([e4m3_lib(c) for c in range(256)])
    S8, _, _ = o.fp8_gemm(p["A"].numpy(), p["B"].numpy(), 2.0, 0.5, 3.0, bias=bias, gamma=gamma)
    ref8 = ((dec[p["A"].numpy()] @ dec[p["B"].numpy()].T) * 3.0 + bias.astype(np.float64)[None, :]) \
        * gamma.astype(np.float64)[:, None]
    assert np.allclose(S8, ref8, rtol=1e-15, atol=0)


def pin_scatter_permutation(o):
    # Scatter by a permutation, then gather back by the same permutation,
    # gives the logical rows; dropped rows keep the prefill.
    D = np.arange(7 * 3, dtype=np.uint16).reshape(7, 3)
    perm = np.random.default_rng(2).permutation(7)
    out = o.scatter_rows(D, perm, np.zeros((7, 3), np.uint16))
    assert np.array_equal(out[perm], D)
    drop = perm.copy()
    drop[[1, 4]] = -1
    out2 = o.scatter_rows(D, drop, np.full((7, 3), 999, np.uint16))
    kept = drop >= 0
    assert np.array_equal(out2[drop[kept]], D[kept])
    assert (np.delete(out2, drop[kept], axis=0) == 999).all()


def pin_grouped_worked(o):
    """tests/golden/nvfp4_grouped_case.txt: two slices with their own
    right-hand sides, without and with bias / gamma (values exact)."""
    g = {}
    for t in _rows("nvfp4_grouped_case.txt"):
        g.setdefault(t[0], []).append(t[1:])
    offs = [int(v) for v in g["offs"][0]]
    row = lambda c: [int(c, 16)] * 16  # noqa: E731
    A = pack(np.array([row(c) for c in g["acodes"][0]], np.uint8))
    B = np.stack([pack(np.array([row(c) for c in g[f"b{e}codes"][0]], np.uint8)) for e in (0, 1)])
    M, N = A.shape[0], B.shape[1]
    sfA = np.full((M, 1), 0x38, np.uint8)
    sfB = np.full((2, N, 1), 0x38, np.uint8)
    alpha = float(g["alpha"][0][0])
    S, T, D = o.nvfp4_grouped_gemm(A, sfA, B, sfB, offs, alpha, 16)
    for r in g["plain"]:
        assert S[int(r[0])].tolist() == [float(v) for v in r[1:]], ("plain", r[0], S[int(r[0])])
    assert np.array_equal(T, np.abs(S))      # every product of a row has one sign
    bias = np.array([[float(v) for v in g["bias0"][0]], [float(v) for v in g["bias1"][0]]], np.float32)
    gamma = np.array([float(v) for v in g["gamma"][0]], np.float32)
    S, _, D = o.nvfp4_grouped_gemm(A, sfA, B, sfB, offs, alpha, 16, bias=bias, gamma=gamma)
    for r in g["D"]:
        want = [float(v) for v in r[1:]]
        assert S[int(r[0])].tolist() == want and oracle.bf16_bits_to_float(D[int(r[0])]).tolist() == want, r[0]


def pin_grouped_single_slice_is_plain(o):
    # E = 1: one slice covering every row is exactly the ordinary GEMM
    M, N, K = 40, 24, 64
    A, sfA, B, sfB = _uniform_problem(M, N, K, 17)
    S0, T0, D0 = o.nvfp4_gemm(A, sfA, B, sfB, 0.625, K)
    S1, T1, D1 = o.nvfp4_grouped_gemm(A, sfA, B[None], sfB[None], [0, M], 0.625, K)
    assert np.array_equal(S0, S1) and np.array_equal(T0, T1) and np.array_equal(D0, D1)


def pin_grouped_numpy(o):
    # Independent restatement over ragged slices (one empty): dequantise
    # with the golden table and the library E4M3 decoder, multiply each
    # slice by its own right-hand side in float64, add that slice's bias,
    # scale rows by gamma. 2^u scales: every sum exact.
    M, N, K, E = 45, 16, 64, 4
    offs = [0, 7, 7, 30, 45]
    A, sfA, _, _ = _uniform_problem(M, N, K, 23)
    Bs, sBs = zip(*[_uniform_problem(M, N, K, 40 + e)[2:] for e in range(E)])
    B, sfB = np.stack(Bs), np.stack(sBs)
    rng = np.random.default_rng(8)
    bias = rng.standard_normal((E, N)).astype(np.float32)
    gamma = rng.standard_normal(M).astype(np.float32)
    S, T, _ = o.nvfp4_grouped_gemm(A, sfA, B, sfB, offs, 1.5, K, bias=bias, gamma=gamma)
    da = deq_nvfp4(A, sfA)
    ref = np.empty((M, N))
    for e in range(E):
        r0, r1 = offs[e], offs[e + 1]
        ref[r0:r1] = (1.5 * (da[r0:r1] @ deq_nvfp4(B[e], sfB[e]).T) + bias[e].astype(np.float64)) \
            * gamma[r0:r1, None].astype(np.float64)
    assert np.allclose(S, ref, rtol=1e-15, atol=0)
    with pytest.raises(ValueError):
        o.nvfp4_grouped_gemm(A, sfA, B, sfB, [0, 7, 6, 30, 45], 1.5, K)    # decreasing offsets


def pin_grouped_scale_layout(o):
    # Each slice is swizzled on its own and starts a new 128-row block row:
    # the byte of (row, col) of slice e sits in block row
    # blk0(e) + (row - offs[e]) // 128, written out here from the layout's
    # definition (row r, column c of a 128 x 4 block at (r%32)*16 + (r//32)*4
    # + c%4, blocks column-block fastest), padding zero.
    K, offs = 96, [0, 130, 130, 200]
    M, cols = offs[-1], K // 16
    ncb = (cols + 3) // 4
    sf = np.random.default_rng(3).integers(1, 256, (M, cols)).astype(np.uint8)
    got = o.swizzle_scales_grouped(sf, offs, K)
    assert got.size == (-(-M // 128) + 3) * 128 * ncb * 4
    want = np.zeros_like(got)
    brow = 0
    for e in range(3):
        for r in range(offs[e], offs[e + 1]):
            lr = r - offs[e]
            for c in range(cols):
                blk = (brow + lr // 128) * ncb + c // 4
                rr = lr % 128
                want[blk * 512 + (rr % 32) * 16 + (rr // 32) * 4 + c % 4] = sf[r, c]
        brow += -(-(offs[e + 1] - offs[e]) // 128)
    assert np.array_equal(got, want)
    # hand-worked landmarks: slice 2 (rows 130..199) starts at block row 2
    # (slice 0 fills two block rows, slice 1 none): its first row's scale 0 is
    # byte 2 * ncb * 512; row 199 (local 69: 69 % 32 = 5, 69 // 32 = 2),
    # scale 5 (column block 1, c % 4 = 1) is byte (2*ncb + 1)*512 + 5*16 + 2*4 + 1.
    assert got[2 * ncb * 512] == sf[130, 0]
    assert got[(2 * ncb + 1) * 512 + 5 * 16 + 2 * 4 + 1] == sf[199, 5]


def pin_dense_worked(o):
    """tests/golden/nvfp4_dense_case.txt: block-scaled E2M1 A times BF16 B."""
    want = {int(r[1]): [float(v) for v in r[2:]] for r in _rows("nvfp4_dense_case.txt") if r[0] == "D"}
    A = pack(np.array([[0x2] * 32, [k % 8 for k in range(32)]], np.uint8))
    sfA = np.array([[0x40, 0x30], [0x38, 0x38]], np.uint8)
    B = _bf16_bits([[0.25] * 16 + [-3.0] * 16, [1.5] * 32])
    S, _, D = o.nvfp4_dense_gemm(A, sfA, B, 1.0, 32)
    for i, row in want.items():
        assert S[i].tolist() == row and oracle.bf16_bits_to_float(D[i]).tolist() == row, (i, S[i])


def pin_dense_reduces_to_nvfp4(o):
    # B's BF16 values exactly the E2M1 values of packed codes with unit
    # scales: the dense GEMM is then the (pinned) NVFP4 GEMM with B's scales
    # all 1.0, bit for bit.
    M, N, K = 24, 40, 128
    A, sfA, Bp, _ = _uniform_problem(M, N, K, 31)
    codes = np.empty((N, K), np.uint8)
    codes[:, 0::2], codes[:, 1::2] = Bp & 15, Bp >> 4
    B_bf16 = _bf16_bits(np.array([E2M1_TABLE[c] for c in codes.reshape(-1)]).reshape(N, K))
    ones = np.full((N, K // 16), 0x38, np.uint8)
    S0, T0, D0 = o.nvfp4_gemm(A, sfA, Bp, ones, 0.75, K)
    S1, T1, D1 = o.nvfp4_dense_gemm(A, sfA, B_bf16, 0.75, K)
    assert np.array_equal(S0, S1) and np.array_equal(T0, T1) and np.array_equal(D0, D1)


def pin_dense_numpy(o):
    # Independent restatement: dequantised A (golden table, library E4M3)
    # times the BF16 values of B (widened by bit shift), numpy float64.
    M, N, K = 20, 36, 256
    A, sfA, _, _ = _uniform_problem(M, N, K, 33)
    B = _random_bf16(N, K, 34)
    S, T, _ = o.nvfp4_dense_gemm(A, sfA, B, 1.25, K)
    bv = _bits_to_f32(B).astype(np.float64)
    ref = 1.25 * (deq_nvfp4(A, sfA) @ bv.T)
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(T, 1.25 * (np.abs(deq_nvfp4(A, sfA)) @ np.abs(bv).T), rtol=1e-12)
    rows, cols = [19, 0, 7], [35, 2]
    S2, _, _ = o.nvfp4_dense_gemm(A, sfA, B, 1.25, K, rows=rows, cols=cols)
    assert np.array_equal(S2, S[np.ix_(rows, cols)])


def pin_dense_f16_worked(o):
    """tests/golden/nvfp4_dense_f16_case.txt: block-scaled E2M1 A times FP16
    B, with a value BF16 cannot hold, the smallest subnormal and the largest
    finite FP16 value."""
    rows = _rows("nvfp4_dense_f16_case.txt")
    bsrc = {int(r[1]): (int(r[2], 16), int(r[3], 16)) for r in rows if r[0] == "B"}
    B = np.array([[bsrc[n][0]] * 16 + [bsrc[n][1]] * 16 for n in (0, 1)], np.uint16)
    A = pack(np.array([[0x2] * 16 + [0x9] * 16], np.uint8))
    sfA = np.array([[0x38, 0x48]], np.uint8)
    S, _, D = o.nvfp4_dense_gemm(A, sfA, B, 1.0, 32, b_f16=True)
    for r in rows:
        if r[0] == "S":
            assert S[int(r[1])].tolist() == [float(v) for v in r[2:]], S
        elif r[0] == "D":
            assert oracle.bf16_bits_to_float(D[int(r[1])]).tolist() == [float(v) for v in r[2:]], D


def _random_f16_bits(rows, K, seed):
    """Random finite IEEE binary16 bit patterns over the whole range
    (normal and subnormal, both signs; exponent field 31 left out)."""
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 1 << 16, (rows, K), dtype=np.uint32).astype(np.uint16)
    inf_nan = (bits & 0x7C00) == 0x7C00
    bits[inf_nan] ^= 0x4000
    return bits


def pin_dense_f16_numpy(o):
    # Independent restatement: dequantised A times B decoded by numpy's own
    # float16 type, in float64; and FP16 B holding the same values as a
    # BF16 B (E2M1 values fit both) gives the BF16 result bit for bit.
    M, N, K = 12, 24, 128
    A, sfA, Bp, _ = _uniform_problem(M, N, K, 35)
    B = _random_f16_bits(N, K, 36)
    S, T, _ = o.nvfp4_dense_gemm(A, sfA, B, 0.5, K, b_f16=True)
    bv = B.view(np.float16).astype(np.float64)
    ref = 0.5 * (deq_nvfp4(A, sfA) @ bv.T)
    assert np.allclose(S, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    assert np.allclose(T, 0.5 * (np.abs(deq_nvfp4(A, sfA)) @ np.abs(bv).T), rtol=1e-12)
    codes = np.empty((N, K), np.uint8)
    codes[:, 0::2], codes[:, 1::2] = Bp & 15, Bp >> 4
    vals = np.array([E2M1_TABLE[c] for c in codes.reshape(-1)]).reshape(N, K)
    got = o.nvfp4_dense_gemm(A, sfA, vals.astype(np.float16).view(np.uint16), 0.5, K, b_f16=True)
    want = o.nvfp4_dense_gemm(A, sfA, _bf16_bits(vals), 0.5, K)
    assert all(np.array_equal(g, w) for g, w in zip(got, want))


def pin_dense_grouped_worked(o):
    """tests/golden/nvfp4_dense_grouped_case.txt: two slices, per-slice
    right-hand side and bias."""
    want = {int(r[1]): [float(v) for v in r[2:]] for r in _rows("nvfp4_dense_grouped_case.txt") if r[0] == "D"}
    rows = np.array([[0x2] * 32, [k % 8 for k in range(32)], [0x2] * 32], np.uint8)
    A = pack(rows)
    sfA = np.array([[0x40, 0x30], [0x38, 0x38], [0x40, 0x30]], np.uint8)
    b0 = [[0.25] * 16 + [-3.0] * 16, [1.5] * 32]
    B = np.stack([_bf16_bits(b0), _bf16_bits(b0[::-1])])
    bias = np.array([[1, 2], [10, 20]], np.float32)
    S, _, D = o.nvfp4_dense_grouped_gemm(A, sfA, B, [0, 2, 3], 1.0, 32, bias=bias)
    for i, row in want.items():
        assert S[i].tolist() == row and oracle.bf16_bits_to_float(D[i]).tolist() == row, (i, S[i])


def pin_dense_grouped_numpy(o):
    # Independent restatement over ragged slices (one empty), both 16-bit
    # right-hand-side types: dequantised A rows of slice e times B[e]'s
    # values, plus bias[e], times the rows' gamma; E = 1 is the plain GEMM.
    M, N, K = 21, 16, 128
    A, sfA, _, _ = _uniform_problem(M, N, K, 37)
    offs = [0, 5, 5, 13, 21]
    E = len(offs) - 1
    rng = np.random.default_rng(38)
    bias = rng.standard_normal((E, N)).astype(np.float32)
    gamma = rng.standard_normal(M).astype(np.float32)
    deq = deq_nvfp4(A, sfA)
    for f16 in (False, True):
        if f16:
            B = np.stack([_random_f16_bits(N, K, 39 + e) for e in range(E)])
            bv = B.view(np.float16).astype(np.float64)
        else:
            B = np.stack([_random_bf16(N, K, 39 + e) for e in range(E)])
            bv = _bits_to_f32(B).astype(np.float64)
        S, _, _ = o.nvfp4_dense_grouped_gemm(A, sfA, B, offs, 0.75, K, bias=bias, gamma=gamma, b_f16=f16)
        ref = np.zeros((M, N))
        for e in range(E):
            r = slice(offs[e], offs[e + 1])
            ref[r] = gamma[r, None].astype(np.float64) * (0.75 * (deq[r] @ bv[e].T) + bias[e].astype(np.float64))
        assert np.allclose(S, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max()), f16
        S1, T1, D1 = o.nvfp4_dense_grouped_gemm(A, sfA, B[:1], [0, M], 0.75, K, b_f16=f16)
        S0, T0, D0 = o.nvfp4_dense_gemm(A, sfA, B[0], 0.75, K, b_f16=f16)
        assert np.array_equal(S1, S0) and np.array_equal(T1, T0) and np.array_equal(D1, D0)


def pin_dense_kragged_worked(o):
    """tests/golden/nvfp4_dense_kragged_case.txt: two slices of K, each its
    own output, the second with a bias row."""
    want = {(int(r[1]), int(r[2])): [float(v) for v in r[3:]] for r in _rows("nvfp4_dense_kragged_case.txt")
            if r[0] == "D"}
    A = pack(np.array([[0x2] * 32, [k % 8 for k in range(32)]], np.uint8))
    sfA = np.array([[0x40, 0x30], [0x38, 0x38]], np.uint8)
    B = _bf16_bits([[0.25] * 16 + [-3.0] * 16, [1.5] * 32])
    bias = np.array([[0, 0], [100, 0]], np.float32)
    S, _, D = o.nvfp4_dense_kgrouped_gemm(A, sfA, B, [0, 16, 32], 1.0, 32, bias=bias)
    for (e, i), row in want.items():
        assert S[e, i].tolist() == row and oracle.bf16_bits_to_float(D[e, i]).tolist() == row, (e, i, S[e, i])


def pin_dense_kragged_partition(o):
    # The slices' sums partition the whole contraction: without bias the
    # unrounded sums over any split of K (an empty slice included) add up
    # to the plain GEMM's, exactly in double for these short sums; and a
    # numpy restatement of each slice in both 16-bit types.
    M, N, K = 9, 16, 256
    A, sfA, _, _ = _uniform_problem(M, N, K, 41)
    deq = deq_nvfp4(A, sfA)
    koffs = [0, 48, 48, 160, 256]
    gamma = np.random.default_rng(42).standard_normal(M).astype(np.float32)
    for f16 in (False, True):
        B = _random_f16_bits(N, K, 43) if f16 else _random_bf16(N, K, 43)
        bv = B.view(np.float16).astype(np.float64) if f16 else _bits_to_f32(B).astype(np.float64)
        S, T, _ = o.nvfp4_dense_kgrouped_gemm(A, sfA, B, koffs, 0.5, K, b_f16=f16)
        S0, T0, _ = o.nvfp4_dense_gemm(A, sfA, B, 0.5, K, b_f16=f16)
        assert np.allclose(S.sum(axis=0), S0, rtol=1e-12, atol=1e-12 * np.abs(S0).max()), f16
        assert np.allclose(T.sum(axis=0), T0, rtol=1e-12), f16
        assert not S[1].any()                                    # the empty slice
        Sg, _, _ = o.nvfp4_dense_kgrouped_gemm(A, sfA, B, koffs, 0.5, K, gamma=gamma, b_f16=f16)
        for e in range(len(koffs) - 1):
            k = slice(koffs[e], koffs[e + 1])
            ref = gamma[:, None].astype(np.float64) * (0.5 * (deq[:, k] @ bv[:, k].T))
            assert np.allclose(Sg[e], ref, rtol=1e-12, atol=1e-12 * max(np.abs(ref).max(), 1.0)), (f16, e)


def _swizzle_numpy(sf: np.ndarray, K: int) -> np.ndarray:
    """Independent restatement of the 128x4-blocked scale layout by reshapes."""
    rows, cols = sf.shape
    pr, pc = -(-rows // 128) * 128, -(-cols // 4) * 4
    pad = np.zeros((pr, pc), np.uint8)
    pad[:rows, :cols] = sf
    # (row-block, r1, r0, col-block, c) with row = 128*rb + 32*r1 + r0
    t = pad.reshape(pr // 128, 4, 32, pc // 4, 4)
    # block order (rb, cb); inside a block byte index r0*16 + r1*4 + c
    return t.transpose(0, 3, 2, 1, 4).reshape(-1).copy()


def pin_swizzle(o):
    # hand-worked offsets for rows = 256, K = 512 (32 scale columns, 8 blocks
    # of 4 per row-block): (r, c) -> block (r//128)*8 + c//4, byte
    # (r%32)*16 + ((r%128)//32)*4 + c%4
    rows, K = 256, 512
    sf = np.zeros((rows, K // 16), np.uint8)
    marks = {(0, 0): 0, (33, 5): 533, (130, 10): 5154, (255, 31): 8191, (96, 3): 15}
    for n, (r, c) in enumerate(marks):
        sf[r, c] = n + 1
    out = o.swizzle_scales(sf, K)
    assert out.size == 8192
    for n, ((r, c), off) in enumerate(marks.items()):
        assert out[off] == n + 1, ((r, c), off)
    assert int((out != 0).sum()) == len(marks)
    # ragged shapes: independent reshape restatement, bijection and zero pad
    rng = np.random.default_rng(3)
    for rows, K in ((1, 16), (127, 48), (129, 64), (300, 1040), (256, 256)):
        sf = rng.integers(1, 256, (rows, K // 16)).astype(np.uint8)
        out = o.swizzle_scales(sf, K)
        assert out.size == o.swizzled_scale_bytes(rows, K)
        assert np.array_equal(out, _swizzle_numpy(sf, K)), (rows, K)
        assert int((out != 0).sum()) == sf.size
        assert np.array_equal(np.sort(out[out != 0]), np.sort(sf.reshape(-1)))


# --------------------------------------------------------------------------
# Two-level NVFP4 quantisation
# --------------------------------------------------------------------------

def _bf16_bits(values) -> np.ndarray:
    t = torch.tensor(np.asarray(values, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _bits_to_f32(bits) -> np.ndarray:
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


E4M3_LIB = np.array([e4m3_lib(c) for c in range(0x7F)])      # positive finite codes, library-decoded
E2M1_MAG = np.array([E2M1_TABLE[c] for c in range(8)])       # golden table


def _unpack(packed: np.ndarray) -> np.ndarray:
    out = np.empty((packed.shape[0], packed.shape[1] * 2), np.uint8)
    out[:, 0::2] = packed & 15
    out[:, 1::2] = packed >> 4
    return out


def pin_quantize_worked(o):
    """The hand-worked two-row case of tests/golden/nvfp4_quantize_case.txt."""
    rows = {}
    for t in _rows("nvfp4_quantize_case.txt"):
        rows.setdefault(t[0], []).append(t[1:])
    X = np.zeros((2, 32), np.uint16)
    for r in rows["x"]:
        X[int(r[0])] = _bf16_bits([float(v) for v in r[1:]])
    packed, sf, amax, sg = o.nvfp4_quantize(X)
    for r in rows["packed"]:
        assert [int(b, 16) for b in r[1:]] == packed[int(r[0])].tolist(), ("packed", r[0])
    for r in rows["scales"]:
        assert [int(b, 16) for b in r[1:]] == sf[int(r[0])].tolist(), ("scales", r[0])
    assert float(amax) == float(rows["amax"][0][0]) and float(sg) == float(rows["sg"][0][0])


def _random_bf16(rows, K, seed, scale=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, K)).astype(np.float32) * np.float32(scale)
    return _bf16_bits(x)


def pin_quantize_nearest_bruteforce(o):
    """Every scale is the nearest positive E4M3 value (library-decoded, ties to
    the even code, saturating at 448) to (bmax / 6) * s_g, and every code the
    nearest E2M1 value (golden table, ties to even, saturating at 6) to
    x * s_g / scale -- each quantity computed here in numpy float32."""
    X = _random_bf16(7, 96, 11)
    packed, sf, amax, sg = o.nvfp4_quantize(X)
    x = _bits_to_f32(X)
    assert amax == np.abs(x).max()
    assert sg == np.float32(2688.0) / np.float32(amax)
    codes = _unpack(packed)
    for r in range(x.shape[0]):
        for b in range(x.shape[1] // 16):
            blk = x[r, 16 * b:16 * b + 16]
            sc = (np.float32(np.abs(blk).max()) / np.float32(6.0)) * sg
            d = np.abs(E4M3_LIB - float(min(sc, np.float32(448.0))))
            best = np.flatnonzero(d == d.min())
            want = best[0] if len(best) == 1 else [c for c in best if c % 2 == 0][0]
            assert sf[r, b] == want, (r, b, sc)
            sv = np.float32(E4M3_LIB[sf[r, b]])
            for k in range(16):
                c = int(codes[r, 16 * b + k])
                if sv == 0:
                    assert c == 0
                    continue
                y = (blk[k] * sg) / sv
                dd = np.abs(E2M1_MAG - abs(float(y)))
                cand = np.flatnonzero(dd == dd.min())
                mag = cand[0] if len(cand) == 1 else [m for m in cand if m % 2 == 0][0]
                assert c == (mag | (8 if np.signbit(y) else 0)), (r, b, k, float(y), c)


def pin_quantize_scale_invariance(o):
    """Scaling X by a power of two leaves codes and scales unchanged and
    scales amax by it and s_g by its inverse, exactly."""
    X = _random_bf16(5, 64, 12)
    ref = o.nvfp4_quantize(X)
    for j in (-3, 5):
        Xj = _bf16_bits(_bits_to_f32(X) * np.float32(2.0 ** j))
        got = o.nvfp4_quantize(Xj)
        assert np.array_equal(got[0], ref[0]) and np.array_equal(got[1], ref[1]), j
        assert got[2] == ref[2] * np.float32(2.0 ** j) and got[3] == ref[3] * np.float32(2.0 ** -j), j


def pin_quantize_amax_element(o):
    """The largest |x| of the tensor lands on +-6 with a block scale of 448."""
    X = _random_bf16(4, 80, 13)
    packed, sf, amax, sg = o.nvfp4_quantize(X)
    x = _bits_to_f32(X)
    r, k = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert sf[r, k // 16] == 0x7E
    assert _unpack(packed)[r, k] == (15 if x[r, k] < 0 else 7)


def pin_quantize_dequant_bound(o):
    """Dequantised values e2m1(code) * scale / s_g are within one scale step
    (the E2M1 spacing is at most 2 below 6, saturation adds under 0.5) of x."""
    X = _random_bf16(6, 128, 14, scale=3.0)
    packed, sf, amax, sg = o.nvfp4_quantize(X)
    x = _bits_to_f32(X).astype(np.float64)
    codes = _unpack(packed)
    val = E2M1_MAG[codes & 7] * np.where(codes & 8, -1.0, 1.0)
    sv = E4M3_LIB[sf].repeat(16, axis=1)
    deq = val * sv / float(sg)
    step = sv / float(sg)
    assert np.all(np.abs(deq - x) <= 1.001 * step)


def pin_freivalds_worked(o):
    """Freivalds' right-hand side on the hand-worked 2x2x32 case: D =
    [[96, 54], [-48, -27]] (every B value >= 0, so T = |D|), hence D x for
    x = (1, -1) and (1, 1) is (42, -21) and (150, -75), and sum_j T[i][j] =
    (150, 75) -- values worked by hand, not by the oracle's GEMM."""
    A = pack(np.array([[0x2] * 32, [0xA] * 32], np.uint8))
    B = pack(np.array([[0x4] * 32, [k % 8 for k in range(32)]], np.uint8))
    sfA = np.array([[0x38, 0x40], [0x30, 0x38]], np.uint8)
    sfB = np.array([[0x38, 0x38], [0x38, 0x28]], np.uint8)
    x = np.array([[1, -1], [1, 1]], np.int8)
    r = o.nvfp4_freivalds(A, sfA, B, sfB, 1.0, 32, x)
    assert np.array_equal(r["y"], [[42.0, -21.0], [150.0, -75.0]]), r["y"]
    assert np.array_equal(r["tsum"], [150.0, 75.0]), r["tsum"]
    assert np.all(r["g"] >= np.abs(r["y"]))


def _freivalds_vs_gemm(o, S, T, r, x):
    ref = S @ x.astype(np.float64).T
    assert np.all(np.abs(r["y"] - ref.T) <= 1e-12 * (r["g"] + np.abs(S).sum(axis=1)[None, :])), "y != S x"
    assert np.allclose(r["tsum"], T.sum(axis=1), rtol=1e-12, atol=0), "tsum != sum_j T"
    assert np.all(r["t2"] >= (T * T).sum(axis=1) * (1 - 1e-12)), "t2 below sum_j T^2"


def pin_freivalds_matches_gemm(o):
    """Freivalds' right-hand side y = alpha Adeq (Bdeq^T x) against the
    pinned element-wise oracle's S x, on ragged shapes of both kinds: the
    same product, associated the other way. Also sum_j T = tsum and the
    Cauchy-Schwarz bound t2 >= sum_j T^2."""
    x = oracle.rademacher(3, 136, seed=5)
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=72, N=136, K=512)
    A, sfA, B, sfB = (p[k].numpy() for k in ("A", "sfA", "B", "sfB"))
    S, T, _ = o.nvfp4_gemm(A, sfA, B, sfB, p["alpha"], 512)
    _freivalds_vs_gemm(o, S, T, o.nvfp4_freivalds(A, sfA, B, sfB, p["alpha"], 512, x), x)
    w8 = workloads.WORKLOADS["fp8_8192"]
    q = workloads.make_fp8(w8, "cpu", M=40, N=136, K=96)
    A8, B8 = q["A"].numpy(), q["B"].numpy()
    S8, T8, _ = o.fp8_gemm(A8, B8, q["alpha"], 0.5, 3.0)
    _freivalds_vs_gemm(o, S8, T8, o.fp8_freivalds(A8, B8, q["alpha"], x, 0.5, 3.0), x)


def pin_freivalds_gram(o):
    """With B = A the product is the Gram matrix: S_ii = alpha sum_k adeq_ik^2,
    so t2_i = alpha^2 a2_i b2 must equal S_ii * sum_j S_jj exactly up to
    rounding -- a check of t2's two sums through the pinned GEMM."""
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=48, N=48, K=256)
    A, sfA = p["A"].numpy(), p["sfA"].numpy()
    S, _, _ = o.nvfp4_gemm(A, sfA, A, sfA, 0.75, 256)
    r = o.nvfp4_freivalds(A, sfA, A, sfA, 0.75, 256, oracle.rademacher(1, 48, seed=2))
    d = np.diag(S)
    assert np.allclose(r["t2"], d * d.sum(), rtol=1e-12, atol=0)


PINS = [pin_e2m1_table, pin_e4m3_codes, pin_bf16_cases, pin_worked_1x1x16, pin_worked_2x2x32,
        pin_one_hot, pin_brute_force_k16, pin_scale_linearity, pin_numpy_definition,
        pin_fraction_exact, pin_fp8_numpy, pin_swizzle, pin_quantize_worked,
        pin_quantize_nearest_bruteforce, pin_quantize_scale_invariance, pin_quantize_amax_element,
        pin_quantize_dequant_bound, pin_epilogue_worked, pin_epilogue_numpy, pin_scatter_permutation,
        pin_grouped_worked, pin_grouped_single_slice_is_plain, pin_grouped_numpy, pin_grouped_scale_layout,
        pin_dense_worked, pin_dense_reduces_to_nvfp4, pin_dense_numpy, pin_dense_f16_worked,
        pin_dense_f16_numpy, pin_dense_grouped_worked, pin_dense_grouped_numpy, pin_dense_kragged_worked,
        pin_dense_kragged_partition, pin_freivalds_worked, pin_freivalds_matches_gemm, pin_freivalds_gram]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(oracle.get())


MUTANTS = ["E2M1_BIAS0", "E2M1_NOSIGN", "E4M3_BIAS8", "SWAP_NIBBLES_A", "DROP_SFB",
           "DROP_LAST_BLOCK", "TRANSPOSE_B", "SWIZZLE_ROWMAJOR_BLOCK", "Q_TIES_AWAY", "Q_NO_SG",
           "Q_SWAP_NIBBLES", "Q_E4M3_CEIL", "EPI_GAMMA_FIRST", "EPI_BIAS_BY_ROW",
           "GROUP_SHIFT", "DENSE_DROP_SFA", "F16_BIAS16", "FV_DROP_SFB", "FV_X_REVERSED", "FV_TSUM_SIGNED"]


@pytest.mark.parametrize("mutant", MUTANTS)
def test_planted_mistake_is_caught(mutant):
    bad = oracle.Oracle(defines=(f"BSO_MUTANT_{mutant}",))
    failed = []
    for pin in PINS:
        try:
            pin(bad)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {mutant}"


def _check_pack_layout(got, X, K):
    """Pins of the tile-packed layout for X uint8[200, K/2], K = 768."""
    rows = X.shape[0]
    assert got.size == oracle.packed_operand_bytes(rows, K) == 256 * 384
    # byte (130, 300): row block 1, row 2 of it; k-block 2, byte 44 = chunk 2, 12 in;
    # chunk 2 XOR row 2 = 0: offset ((1 * 3 + 2) * 128 + 2) * 128 + 0 * 16 + 12
    assert got[((1 * 3 + 2) * 128 + 2) * 128 + 12] == X[130, 300]
    # byte (7, 5): tile 0, row 7, chunk 0 XOR 7 = 7: offset 7 * 128 + 7 * 16 + 5
    assert got[7 * 128 + 7 * 16 + 5] == X[7, 5]
    # restatement: pad, split rows into (rb, r) and bytes into (kb, chunk, b),
    # swizzle the chunk index by r % 8, reorder to (rb, kb, r, chunk, b)
    pad = np.zeros((256, K // 2), np.uint8)
    pad[:rows] = X
    t = pad.reshape(2, 128, 3, 8, 16)
    sw = np.empty_like(t)
    for r in range(128):
        sw[:, r, :, np.arange(8) ^ (r % 8), :] = t[:, r, :, :, :].transpose(2, 0, 1, 3)
    want = sw.transpose(0, 2, 1, 3, 4).reshape(-1)
    assert np.array_equal(got, want)
    assert not got[(1 * 3 + 0) * 16384 + 72 * 128:(1 * 3 + 1) * 16384].any()   # rows 200.. of tile (1, 0)


PACK_X = np.random.default_rng(17).integers(0, 256, (200, 384)).astype(np.uint8)


def test_pack_operand_tiles_layout():
    """The tile-packed operand layout against hand-computed offsets and an
    independent restatement by reshapes; padding rows are zero."""
    _check_pack_layout(oracle.pack_operand_tiles(PACK_X, 768), PACK_X, 768)


def _pack_mutant(X, K, kind):
    """A plausible wrong tile layout, written out as the oracle's is."""
    rows, width = X.shape
    kblocks, rblocks = K // 256, -(-rows // 128)
    out = np.zeros(rblocks * 128 * width, np.uint8)
    for r in range(rows):
        rb, rr = divmod(r, 128)
        for c in range(width):
            kb, cc = divmod(c, 128)
            chunk = cc // 16 if kind == "no_swizzle" else (cc // 16) ^ (rr % 8)
            tile = kb * rblocks + rb if kind == "k_major_tiles" else rb * kblocks + kb
            out[(tile * 128 + rr) * 128 + chunk * 16 + cc % 16] = X[r, c]
    if kind == "padding_not_zero":
        out[(1 * kblocks) * 16384 + 100 * 128] = 1
    return out


@pytest.mark.parametrize("kind", ["no_swizzle", "k_major_tiles", "padding_not_zero"])
def test_pack_layout_pins_catch_planted_mistakes(kind):
    with pytest.raises(AssertionError):
        _check_pack_layout(_pack_mutant(PACK_X, 768, kind), PACK_X, 768)


def test_tolerance_helper():
    b = lambda x: np.array([oracle.get().bf16_rne(v) for v in x], np.uint16)  # noqa: E731
    ref = b([100.0, 0.0, -3.0, 1.0])
    T = np.array([1e4, 2.0 ** 20, 1.0, 1.0])
    # within: one BF16 ulp of 100 (0.5 <= 2^-7 * 100); |0.5| <= 2^-20 * 2^20
    assert oracle.within_tolerance(b([100.5, 0.5, -3.0, 1.0]), ref, T).all()
    # outside: two ulps of 100; 1.5 > 1; wrong sign; NaN
    got = oracle.within_tolerance(b([101.0, 1.5, 3.0, float("nan")]), ref, T)
    assert not got.any()


def test_oracle_row_col_selection_matches_full():
    A, sfA, B, sfB = _uniform_problem(40, 56, 128, 21)
    o = oracle.get()
    S, T, D = o.nvfp4_gemm(A, sfA, B, sfB, 1.5, 128)
    rows, cols = [39, 0, 17], [55, 3]
    S2, T2, D2 = o.nvfp4_gemm(A, sfA, B, sfB, 1.5, 128, rows=rows, cols=cols, nthreads=3)
    assert np.array_equal(S2, S[np.ix_(rows, cols)]) and np.array_equal(D2, D[np.ix_(rows, cols)])
    assert np.array_equal(T2, T[np.ix_(rows, cols)])
    with pytest.raises(ValueError):
        o.nvfp4_gemm(A, sfA, B, sfB, 1.0, 128, rows=[40])
