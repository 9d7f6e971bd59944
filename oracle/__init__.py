"""CPU oracle for the block-scaled GEMM (test infrastructure).

This package is the plain, slow definition the CUDA library is checked
against: ``D = alpha * (A (.) sA)(B (.) sB)^T`` with E2M1 / E4M3 elements
decoded exactly, accumulation in double and one final rounding to BF16; the
scale layout the tensor core reads; and the two-level NVFP4 quantisation
(BF16 -> E2M1 codes + E4M3 block scales + a global scale) in front of it.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import it. The library (``block_scaled_precision_persistent_gb300``)
never does, and this package imports nothing from the library: the two share
no code, header, table or constant.

The arithmetic lives in ``bsgemm_oracle.c`` (plain C, compiled with gcc on
first use); this module only marshals numpy arrays through ctypes.

Sources the definition follows (page title, section):
  * "Together AI Ports ThunderKittens GEMM Kernels to NVIDIA Vera Rubin NVL72",
    introduction and "Building the GEMM" -- NVFP4 / FP8 GEMMs with block
    scaling factors consumed by the tensor-core MMA.
  * "Triton #11171 - Why Two New NVFP4 Test Cases Produced Twelve
    Tensor-Memory Failures", "The matrix also compared Triton with a reference
    implementation" -- comparison against a reference under a
    format-specific tolerance; "Activation-scale swizzling forced the relevant
    persistent path" -- the scale layout rewritten in HBM for the persistent
    kernel.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "bsgemm_oracle.c"
_BUILD = _HERE / "_build"

# Tolerance of the parity check: |D_gpu - D_ref| <= REL * |D_ref| + ABS * T.
REL_TOL = 2.0 ** -7
ABS_TOL = 2.0 ** -20


def build(out: Path | None = None, defines: tuple[str, ...] = ()) -> Path:
    """Compile the oracle with gcc into a shared object and return its path.

    ``defines`` selects planted-mistake variants (``BSO_MUTANT_*``) that the
    negative-control tests use to show each pin can fail.
    """
    if out is None:
        tag = "_".join(d.lower() for d in defines)
        out = _BUILD / (f"liboracle_{tag}.so" if tag else "liboracle.so")
    out = Path(out)
    if out.exists() and out.stat().st_mtime >= _SRC.stat().st_mtime:
        return out
    out.parent.mkdir(parents=True, exist_ok=True)
    tmp = out.with_suffix(f".tmp{os.getpid()}.so")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-ffp-contract=off", "-fno-fast-math",
           "-fPIC", "-shared", "-pthread", "-o", str(tmp), str(_SRC), "-lm"]
    cmd[1:1] = [f"-D{d}" for d in defines]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """ctypes view of one compiled oracle (the real one or a planted variant)."""

    def __init__(self, defines: tuple[str, ...] = ()):
        self.lib = ctypes.CDLL(str(build(defines=defines)))
        L = self.lib
        u8p = ctypes.POINTER(ctypes.c_uint8)
        i32p = ctypes.POINTER(ctypes.c_int32)
        f64p = ctypes.POINTER(ctypes.c_double)
        u16p = ctypes.POINTER(ctypes.c_uint16)
        L.bso_e2m1.restype = ctypes.c_double
        L.bso_e2m1.argtypes = [ctypes.c_uint]
        L.bso_e4m3.restype = ctypes.c_double
        L.bso_e4m3.argtypes = [ctypes.c_uint]
        L.bso_bf16_rne.restype = ctypes.c_uint16
        L.bso_bf16_rne.argtypes = [ctypes.c_double]
        L.bso_nvfp4_gemm.restype = ctypes.c_int
        f32p = ctypes.POINTER(ctypes.c_float)
        L.bso_nvfp4_gemm.argtypes = [ctypes.c_int] * 3 + [u8p] * 4 + [ctypes.c_float, f32p, f32p,
                                    i32p, ctypes.c_int, i32p, ctypes.c_int, f64p, f64p, u16p,
                                    ctypes.c_int]
        L.bso_fp8_gemm.restype = ctypes.c_int
        L.bso_fp8_gemm.argtypes = [ctypes.c_int] * 3 + [u8p] * 2 + [ctypes.c_float] * 3 + [
            f32p, f32p, i32p, ctypes.c_int, i32p, ctypes.c_int, f64p, f64p, u16p, ctypes.c_int]
        L.bso_swizzled_scale_bytes.restype = ctypes.c_size_t
        L.bso_swizzled_scale_bytes.argtypes = [ctypes.c_int, ctypes.c_int]
        L.bso_swizzle_scales.restype = ctypes.c_int
        L.bso_swizzle_scales.argtypes = [ctypes.c_int, ctypes.c_int, u8p, u8p]
        L.bso_nvfp4_dense_gemm.restype = ctypes.c_int
        L.bso_nvfp4_dense_gemm.argtypes = [ctypes.c_int] * 3 + [u8p, u8p, u16p, ctypes.c_int, ctypes.c_float, f32p, f32p,
                                                                i32p, ctypes.c_int, i32p, ctypes.c_int, f64p, f64p,
                                                                u16p, ctypes.c_int]
        L.bso_nvfp4_grouped_gemm.restype = ctypes.c_int
        L.bso_nvfp4_grouped_gemm.argtypes = [ctypes.c_int] * 4 + [u8p] * 4 + [i32p, ctypes.c_float, f32p, f32p,
                                                                         f64p, f64p, u16p, ctypes.c_int]
        L.bso_grouped_scale_bytes.restype = ctypes.c_size_t
        L.bso_grouped_scale_bytes.argtypes = [ctypes.c_int] * 3
        L.bso_swizzle_scales_grouped.restype = ctypes.c_int
        L.bso_swizzle_scales_grouped.argtypes = [ctypes.c_int] * 3 + [i32p, u8p, u8p]
        i8p = ctypes.POINTER(ctypes.c_int8)
        L.bso_nvfp4_freivalds.restype = ctypes.c_int
        L.bso_nvfp4_freivalds.argtypes = [ctypes.c_int] * 3 + [u8p] * 4 + [ctypes.c_float, i8p, ctypes.c_int] + [
            f64p] * 4 + [ctypes.c_int]
        L.bso_fp8_freivalds.restype = ctypes.c_int
        L.bso_fp8_freivalds.argtypes = [ctypes.c_int] * 3 + [u8p] * 2 + [ctypes.c_float] * 3 + [
            i8p, ctypes.c_int] + [f64p] * 4 + [ctypes.c_int]
        L.bso_nvfp4_quantize.restype = ctypes.c_int
        L.bso_nvfp4_quantize.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_uint16),
                                         u8p, u8p, ctypes.POINTER(ctypes.c_float),
                                         ctypes.POINTER(ctypes.c_float)]

    # -- element decoders -------------------------------------------------
    def e2m1(self, code: int) -> float:
        return self.lib.bso_e2m1(code)

    def e4m3(self, code: int) -> float:
        return self.lib.bso_e4m3(code)

    def bf16_rne(self, x: float) -> int:
        return int(self.lib.bso_bf16_rne(float(x)))

    # -- GEMMs --------------------------------------------------------------
    @staticmethod
    def _sel(sel, lim):
        if sel is None:
            return None, lim
        arr = np.ascontiguousarray(np.asarray(sel, dtype=np.int32))
        return arr, int(arr.size)

    @staticmethod
    def _p(a, ct):
        return None if a is None else a.ctypes.data_as(ctypes.POINTER(ct))

    @staticmethod
    def _vec(v, n):
        if v is None:
            return None
        arr = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
        assert arr.shape == (n,), (arr.shape, n)
        return arr

    def nvfp4_gemm(self, A, sfA, B, sfB, alpha, K, rows=None, cols=None, nthreads=None,
                   bias=None, gamma=None):
        """Return (S, T, D_bits) over the selected rows x cols.

        A: uint8[M, K/2], sfA: uint8[M, K/16], B: uint8[N, K/2], sfB: uint8[N, K/16].
        bias: float32[N] or None, gamma: float32[M] or None (the epilogue
        S' = gamma[i] * (S + bias[j])). S is the unrounded double result, T the
        magnitude sum of the tolerance, D_bits the BF16 bit patterns (uint16)
        of S rounded once. Rows come in logical (computed) order; see
        scatter_rows for the scattered output placement.
        """
        A = np.ascontiguousarray(A, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
        sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
        M, N = A.shape[0], B.shape[0]
        assert A.shape == (M, K // 2) and B.shape == (N, K // 2)
        assert sfA.shape == (M, K // 16) and sfB.shape == (N, K // 16)
        bias, gamma = self._vec(bias, N), self._vec(gamma, M)
        r, nr = self._sel(rows, M)
        c, nc = self._sel(cols, N)
        S = np.empty((nr, nc), np.float64)
        T = np.empty((nr, nc), np.float64)
        D = np.empty((nr, nc), np.uint16)
        rc = self.lib.bso_nvfp4_gemm(M, N, K, self._p(A, ctypes.c_uint8), self._p(sfA, ctypes.c_uint8),
                                     self._p(B, ctypes.c_uint8), self._p(sfB, ctypes.c_uint8),
                                     float(alpha), self._p(bias, ctypes.c_float),
                                     self._p(gamma, ctypes.c_float), self._p(r, ctypes.c_int32), nr,
                                     self._p(c, ctypes.c_int32), nc, self._p(S, ctypes.c_double),
                                     self._p(T, ctypes.c_double), self._p(D, ctypes.c_uint16),
                                     nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"bso_nvfp4_gemm rejected its arguments (rc={rc})")
        return S, T, D

    def fp8_gemm(self, A, B, alpha, sA=1.0, sB=1.0, rows=None, cols=None, nthreads=None,
                 bias=None, gamma=None):
        """FP8 E4M3 GEMM: D = alpha*sA*sB * A B^T. A: uint8[M, K], B: uint8[N, K];
        bias / gamma as for nvfp4_gemm."""
        A = np.ascontiguousarray(A, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        M, K = A.shape
        N = B.shape[0]
        assert B.shape == (N, K)
        bias, gamma = self._vec(bias, N), self._vec(gamma, M)
        r, nr = self._sel(rows, M)
        c, nc = self._sel(cols, N)
        S = np.empty((nr, nc), np.float64)
        T = np.empty((nr, nc), np.float64)
        D = np.empty((nr, nc), np.uint16)
        rc = self.lib.bso_fp8_gemm(M, N, K, self._p(A, ctypes.c_uint8), self._p(B, ctypes.c_uint8),
                                   float(alpha), float(sA), float(sB), self._p(bias, ctypes.c_float),
                                   self._p(gamma, ctypes.c_float), self._p(r, ctypes.c_int32), nr,
                                   self._p(c, ctypes.c_int32), nc, self._p(S, ctypes.c_double),
                                   self._p(T, ctypes.c_double), self._p(D, ctypes.c_uint16),
                                   nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"bso_fp8_gemm rejected its arguments (rc={rc})")
        return S, T, D

    def nvfp4_dense_gemm(self, A, sfA, B_bits, alpha, K, rows=None, cols=None, nthreads=None,
                         bias=None, gamma=None, b_f16=False):
        """NVFP4 x dense GEMM: A uint8[M, K/2] with sfA uint8[M, K/16], B
        uint16[N, K] bit patterns of BF16 (default) or FP16 (b_f16) values.
        Returns (S, T, D_bits) over the selected rows x cols, with the
        epilogue of nvfp4_gemm."""
        B_bf16_bits = B_bits
        A = np.ascontiguousarray(A, dtype=np.uint8)
        sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
        B = np.ascontiguousarray(B_bf16_bits, dtype=np.uint16)
        M, N = A.shape[0], B.shape[0]
        assert A.shape == (M, K // 2) and sfA.shape == (M, K // 16) and B.shape == (N, K)
        bias, gamma = self._vec(bias, N), self._vec(gamma, M)
        r, nr = self._sel(rows, M)
        c, nc = self._sel(cols, N)
        S = np.empty((nr, nc), np.float64)
        T = np.empty((nr, nc), np.float64)
        D = np.empty((nr, nc), np.uint16)
        rc = self.lib.bso_nvfp4_dense_gemm(M, N, K, self._p(A, ctypes.c_uint8), self._p(sfA, ctypes.c_uint8),
                                           self._p(B, ctypes.c_uint16), 1 if b_f16 else 0, float(alpha),
                                           self._p(bias, ctypes.c_float),
                                           self._p(gamma, ctypes.c_float), self._p(r, ctypes.c_int32), nr,
                                           self._p(c, ctypes.c_int32), nc, self._p(S, ctypes.c_double),
                                           self._p(T, ctypes.c_double), self._p(D, ctypes.c_uint16),
                                           nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"bso_nvfp4_dense_gemm rejected its arguments (rc={rc})")
        return S, T, D

    def nvfp4_grouped_gemm(self, A, sfA, B, sfB, offs, alpha, K, bias=None, gamma=None, nthreads=None):
        """Grouped (ragged) NVFP4 GEMM: rows [offs[e], offs[e+1]) of A times
        B[e]^T for each slice e. A: uint8[M, K/2], sfA: uint8[M, K/16],
        B: uint8[E, N, K/2], sfB: uint8[E, N, K/16], offs: int32[E+1],
        bias: float32[E, N] or None, gamma: float32[M] or None.
        Returns (S, T, D_bits), each [M, N] in row order."""
        A = np.ascontiguousarray(A, dtype=np.uint8)
        sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
        offs = np.ascontiguousarray(offs, dtype=np.int32)
        E, N = B.shape[0], B.shape[1]
        M = A.shape[0]
        assert B.shape == (E, N, K // 2) and sfB.shape == (E, N, K // 16) and offs.shape == (E + 1,)
        assert A.shape == (M, K // 2) and sfA.shape == (M, K // 16)
        if bias is not None:
            bias = np.ascontiguousarray(np.asarray(bias, dtype=np.float32))
            assert bias.shape == (E, N)
        gamma = self._vec(gamma, M)
        S = np.empty((M, N), np.float64)
        T = np.empty((M, N), np.float64)
        D = np.empty((M, N), np.uint16)
        rc = self.lib.bso_nvfp4_grouped_gemm(E, M, N, K, self._p(A, ctypes.c_uint8), self._p(sfA, ctypes.c_uint8),
                                             self._p(B, ctypes.c_uint8), self._p(sfB, ctypes.c_uint8),
                                             self._p(offs, ctypes.c_int32), float(alpha),
                                             self._p(bias, ctypes.c_float), self._p(gamma, ctypes.c_float),
                                             self._p(S, ctypes.c_double), self._p(T, ctypes.c_double),
                                             self._p(D, ctypes.c_uint16), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"bso_nvfp4_grouped_gemm rejected its arguments (rc={rc})")
        return S, T, D

    def nvfp4_dense_grouped_gemm(self, A, sfA, B_bits, offs, alpha, K, bias=None, gamma=None, b_f16=False,
                                 nthreads=None):
        """Grouped (routed) NVFP4 x dense GEMM ("Triton #11171 - Why Two New
        NVFP4 Test Cases Produced Twelve Tensor-Memory Failures", section
        "Ragged mode added routing rather than a plain matrix", with the
        dense BF16 / FP16 right-hand side of the opening): rows
        [offs[e], offs[e+1]) of A times B_bits[e]^T for each slice e, each
        slice exactly nvfp4_dense_gemm on its own rows with bias[e] and its
        rows' gamma. A: uint8[M, K/2], sfA: uint8[M, K/16] row-major,
        B_bits: uint16[E, N, K] (BF16, or FP16 with b_f16), offs: int32[E+1]
        with offs[0] = 0, nondecreasing, offs[E] = M; bias: float32[E, N] or
        None; gamma: float32[M] or None. Returns (S, T, D_bits), [M, N]."""
        A = np.ascontiguousarray(A, dtype=np.uint8)
        sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
        B = np.ascontiguousarray(B_bits, dtype=np.uint16)
        offs = [int(v) for v in np.asarray(offs).reshape(-1)]
        E, N, M = B.shape[0], B.shape[1], A.shape[0]
        assert B.shape == (E, N, K) and len(offs) == E + 1
        if offs[0] != 0 or offs[E] != M or any(offs[e] > offs[e + 1] for e in range(E)):
            raise ValueError("offs must start at 0, not decrease, and end at M")
        if bias is not None:
            bias = np.asarray(bias, dtype=np.float32)
            assert bias.shape == (E, N)
        gamma = None if gamma is None else np.asarray(gamma, dtype=np.float32).reshape(M)
        S = np.zeros((M, N), np.float64)
        T = np.zeros((M, N), np.float64)
        D = np.zeros((M, N), np.uint16)
        for e in range(E):
            r0, r1 = offs[e], offs[e + 1]
            if r1 == r0:
                continue
            S[r0:r1], T[r0:r1], D[r0:r1] = self.nvfp4_dense_gemm(
                A[r0:r1], sfA[r0:r1], B[e], alpha, K, nthreads=nthreads,
                bias=None if bias is None else bias[e], gamma=None if gamma is None else gamma[r0:r1], b_f16=b_f16)
        return S, T, D

    def nvfp4_dense_kgrouped_gemm(self, A, sfA, B_bits, koffs, alpha, K, bias=None, gamma=None, b_f16=False,
                                  nthreads=None):
        """Inner-expert (K-ragged) NVFP4 x dense GEMM ("Triton #11171 - Why
        Two New NVFP4 Test Cases Produced Twelve Tensor-Memory Failures",
        section "Why `pad_a` represents the K-ragged boundary": the ragged
        dimension is A's K, padded per slice): K is split into E slices at
        koffs, and slice e gives its own output
            D[e] = epilogue( alpha * A[:, K_e] (x) sA  .  B[:, K_e]^T )
        with bias[e] and gamma -- each slice exactly nvfp4_dense_gemm on its
        columns. koffs: koffs[0] = 0, nondecreasing, koffs[E] = K, every one
        a multiple of 16 (a whole scale block). An empty slice sums nothing.
        A: uint8[M, K/2], sfA: uint8[M, K/16], B_bits: uint16[N, K] (BF16, or
        FP16 with b_f16). Returns (S, T, D_bits), each [E, M, N]."""
        A = np.ascontiguousarray(A, dtype=np.uint8)
        sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
        B = np.ascontiguousarray(B_bits, dtype=np.uint16)
        koffs = [int(v) for v in np.asarray(koffs).reshape(-1)]
        E, M, N = len(koffs) - 1, A.shape[0], B.shape[0]
        assert A.shape == (M, K // 2) and sfA.shape == (M, K // 16) and B.shape == (N, K)
        if koffs[0] != 0 or koffs[E] != K or any(koffs[e] > koffs[e + 1] or koffs[e] % 16 for e in range(E)):
            raise ValueError("koffs must start at 0, not decrease, end at K and fall on 16-element blocks")
        if bias is not None:
            bias = np.asarray(bias, dtype=np.float32)
            assert bias.shape == (E, N)
        S = np.zeros((E, M, N), np.float64)
        T = np.zeros((E, M, N), np.float64)
        D = np.zeros((E, M, N), np.uint16)
        for e in range(E):
            k0, k1 = koffs[e], koffs[e + 1]
            if k1 > k0:
                a, sa, b, k = A[:, k0 // 2:k1 // 2], sfA[:, k0 // 16:k1 // 16], B[:, k0:k1], k1 - k0
            else:   # an empty slice: one block of zero codes sums to exactly zero
                a, sa, b, k = (np.zeros((M, 8), np.uint8), np.full((M, 1), 0x38, np.uint8),
                               np.zeros((N, 16), np.uint16), 16)
            S[e], T[e], D[e] = self.nvfp4_dense_gemm(a, sa, b, alpha, k, nthreads=nthreads,
                                                     bias=None if bias is None else bias[e], gamma=gamma,
                                                     b_f16=b_f16)
        return S, T, D

    # -- Freivalds' check of a whole product --------------------------------
    def _freivalds_out(self, M, x):
        x = np.ascontiguousarray(x, dtype=np.int8)
        nv = x.shape[0]
        return x, nv, np.empty((nv, M)), np.empty((nv, M)), np.empty(M), np.empty(M)

    def nvfp4_freivalds(self, A, sfA, B, sfB, alpha, K, x, nthreads=None):
        """Right-hand side of Freivalds' check for the NVFP4 GEMM, for the
        int8 vectors x[nv, N]: a dict with y = alpha Adeq (Bdeq^T x_q) and
        its rounding bound g (both [nv, M]), tsum[i] = sum_j T[i][j] and
        t2[i] >= sum_j T[i][j]^2 ([M]); see bso_nvfp4_freivalds."""
        A = np.ascontiguousarray(A, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        sfA = np.ascontiguousarray(sfA, dtype=np.uint8)
        sfB = np.ascontiguousarray(sfB, dtype=np.uint8)
        M, N = A.shape[0], B.shape[0]
        assert A.shape == (M, K // 2) and B.shape == (N, K // 2)
        assert sfA.shape == (M, K // 16) and sfB.shape == (N, K // 16)
        x, nv, y, g, tsum, t2 = self._freivalds_out(M, x)
        assert x.shape == (nv, N)
        rc = self.lib.bso_nvfp4_freivalds(M, N, K, self._p(A, ctypes.c_uint8), self._p(sfA, ctypes.c_uint8),
                                          self._p(B, ctypes.c_uint8), self._p(sfB, ctypes.c_uint8), float(alpha),
                                          self._p(x, ctypes.c_int8), nv, self._p(y, ctypes.c_double),
                                          self._p(g, ctypes.c_double), self._p(tsum, ctypes.c_double),
                                          self._p(t2, ctypes.c_double), nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"bso_nvfp4_freivalds failed (rc={rc})")
        return dict(y=y, g=g, tsum=tsum, t2=t2, K=K)

    def fp8_freivalds(self, A, B, alpha, x, sA=1.0, sB=1.0, nthreads=None):
        """As nvfp4_freivalds, for the FP8 GEMM (A uint8[M, K], B uint8[N, K])."""
        A = np.ascontiguousarray(A, dtype=np.uint8)
        B = np.ascontiguousarray(B, dtype=np.uint8)
        M, K = A.shape
        N = B.shape[0]
        assert B.shape == (N, K)
        x, nv, y, g, tsum, t2 = self._freivalds_out(M, x)
        assert x.shape == (nv, N)
        rc = self.lib.bso_fp8_freivalds(M, N, K, self._p(A, ctypes.c_uint8), self._p(B, ctypes.c_uint8),
                                        float(alpha), float(sA), float(sB), self._p(x, ctypes.c_int8), nv,
                                        self._p(y, ctypes.c_double), self._p(g, ctypes.c_double),
                                        self._p(tsum, ctypes.c_double), self._p(t2, ctypes.c_double),
                                        nthreads or default_threads())
        if rc != 0:
            raise ValueError(f"bso_fp8_freivalds failed (rc={rc})")
        return dict(y=y, g=g, tsum=tsum, t2=t2, K=K)

    def grouped_scale_bytes(self, E: int, M: int, K: int) -> int:
        return int(self.lib.bso_grouped_scale_bytes(E, M, K))

    def swizzle_scales_grouped(self, sf, offs, K: int):
        """Row-major uint8[M, K/16] scales of a grouped A -> the per-slice
        swizzled layout (1-D uint8 of grouped_scale_bytes(E, M, K))."""
        sf = np.ascontiguousarray(sf, dtype=np.uint8)
        offs = np.ascontiguousarray(offs, dtype=np.int32)
        E, M = offs.size - 1, sf.shape[0]
        out = np.empty(self.grouped_scale_bytes(E, M, K), np.uint8)
        rc = self.lib.bso_swizzle_scales_grouped(E, M, K, self._p(offs, ctypes.c_int32),
                                                 self._p(sf, ctypes.c_uint8), self._p(out, ctypes.c_uint8))
        if rc != 0:
            raise ValueError("bso_swizzle_scales_grouped rejected its arguments")
        return out

    @staticmethod
    def scatter_rows(D_rows, scatter, out):
        """Scattered output placement ("Triton #11171 ...", section "Scatter
        changes where output rows are written"): logical computed row i goes to
        physical row scatter[i] of `out` (modified in place and returned). A
        destination outside [0, out rows) writes nothing -- a negative index
        marks a row to drop. Destinations must be distinct."""
        D_rows = np.asarray(D_rows)
        dst = np.asarray(scatter, dtype=np.int64)
        assert dst.shape == (D_rows.shape[0],)
        for i in range(dst.size):
            if 0 <= dst[i] < out.shape[0]:
                out[dst[i]] = D_rows[i]
        return out

    # -- scale layout ---------------------------------------------------------
    def nvfp4_quantize(self, x_bf16_bits):
        """Two-level NVFP4 quantisation of BF16 X (uint16 bit patterns
        [rows, K]) -> (packed uint8[rows, K/2], scales uint8[rows, K/16]
        row-major, amax, s_g) with amax and s_g as float32 values."""
        X = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
        rows, K = X.shape
        packed = np.zeros((rows, K // 2), np.uint8)
        sf = np.zeros((rows, K // 16), np.uint8)
        amax = ctypes.c_float(0.0)
        sg = ctypes.c_float(0.0)
        rc = self.lib.bso_nvfp4_quantize(rows, K, X.ctypes.data_as(ctypes.POINTER(ctypes.c_uint16)),
                                         self._p(packed, ctypes.c_uint8), self._p(sf, ctypes.c_uint8),
                                         ctypes.byref(amax), ctypes.byref(sg))
        if rc != 0:
            raise ValueError(f"bso_nvfp4_quantize: bad arguments ({rows}x{K})")
        return packed, sf, np.float32(amax.value), np.float32(sg.value)

    def swizzled_scale_bytes(self, rows: int, K: int) -> int:
        return int(self.lib.bso_swizzled_scale_bytes(rows, K))

    def swizzle_scales(self, sf, K: int):
        """Row-major uint8[rows, K/16] scales -> the 128x4-blocked layout (1-D uint8)."""
        sf = np.ascontiguousarray(sf, dtype=np.uint8)
        rows = sf.shape[0]
        assert sf.shape == (rows, K // 16)
        out = np.empty(self.swizzled_scale_bytes(rows, K), np.uint8)
        rc = self.lib.bso_swizzle_scales(rows, K, self._p(sf, ctypes.c_uint8),
                                         self._p(out, ctypes.c_uint8))
        if rc != 0:
            raise ValueError("bso_swizzle_scales rejected its arguments")
        return out


def packed_operand_bytes(rows: int, K: int) -> int:
    """Bytes of an NVFP4 operand of `rows` rows in the tile-packed layout:
    rows padded to 128, K / 2 bytes a row (K % 256 == 0)."""
    return -(-rows // 128) * 128 * (K // 2)


def pack_operand_tiles(X, K: int) -> np.ndarray:
    """Tile-packed layout of a row-major NVFP4 operand X uint8[rows, K/2]
    (the library's own format, for copies of whole tiles): tile (rb, kb)
    holds rows 128 rb .. 128 rb + 127 and bytes 128 kb .. 128 kb + 127 of
    each, contiguously at tile index rb * (K / 256) + kb, 16 KiB a tile; in a
    tile, byte c of row r sits at r * 128 + ((c // 16) XOR (r % 8)) * 16 +
    c % 16 (the 128-byte swizzle); rows past the end are zero. Written out
    byte by byte (1-D uint8 of packed_operand_bytes(rows, K))."""
    X = np.ascontiguousarray(X, dtype=np.uint8)
    rows, width = X.shape
    assert K % 256 == 0 and width == K // 2
    kblocks = K // 256
    out = np.zeros(packed_operand_bytes(rows, K), np.uint8)
    for r in range(rows):
        rb, rr = divmod(r, 128)
        for c in range(width):
            kb, cc = divmod(c, 128)
            off = ((rb * kblocks + kb) * 128 + rr) * 128 + ((cc // 16) ^ (rr % 8)) * 16 + cc % 16
            out[off] = X[r, c]
    return out


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


_default: Oracle | None = None


def get() -> Oracle:
    """The real (unplanted) oracle, compiled on first use."""
    global _default
    if _default is None:
        _default = Oracle()
    return _default


def bf16_bits_to_float(bits) -> np.ndarray:
    """Widen BF16 bit patterns (uint16) to float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def within_tolerance(d_gpu_bits, d_ref_bits, T) -> np.ndarray:
    """Element-wise |D_gpu - D_ref| <= 2^-7 |D_ref| + 2^-20 T (both BF16).

    NaN is never within tolerance; +0 and -0 compare equal.
    """
    g = bf16_bits_to_float(d_gpu_bits)
    r = bf16_bits_to_float(d_ref_bits)
    with np.errstate(invalid="ignore"):
        ok = np.abs(g - r) <= REL_TOL * np.abs(r) + ABS_TOL * np.asarray(T, np.float64)
    both_inf = np.isinf(g) & np.isinf(r) & (np.sign(g) == np.sign(r))
    return (ok | both_inf) & ~np.isnan(g) & ~np.isnan(r)


# -- Freivalds' check: the decision ------------------------------------------
#
# R. Freivalds (1977): D x = alpha Adeq (Bdeq^T x) for a correct D and any x.
# The oracle computes the right-hand side y exactly up to one double dot
# product's rounding (Oracle.nvfp4_freivalds / fp8_freivalds); here the left
# side z = D_gpu x is formed from the GPU's BF16 bits and r = z - y is
# compared with what the element-wise tolerance allows.
#
# Per element, D_gpu may differ from the exact value S by
#     |e_ij| <= c1 |D_gpu_ij| + c2 T_ij,
# with rho = 2^-7 + 2^-8 / (1 - 2^-8) (the tolerance against the rounded
# D_ref plus D_ref's own BF16 rounding of S), c1 = rho / (1 - 2^-7) and
# c2 = 2^-20 (1 + c1): D_ref is bounded through D_gpu, which is known.
#
# Two bounds on |r_i| are checked, both must hold:
#   * summed (deterministic): sum_j (c1 |D_ij| + c2 T_ij) |x_j| -- what the
#     element-wise tolerance allows in the worst case; it can never fail for a
#     result that is within tolerance everywhere.
#   * Hoeffding (probabilistic): x has independent +-1 entries drawn
#     independently of D, so P(|sum_j e_ij x_j| >= C s_i) <= 2 exp(-C^2 / 2)
#     with s_i^2 = sum_j e_ij^2 <= (c1 sqrt(sum_j D_ij^2) + c2 sqrt(t2_i))^2
#     (Minkowski). With C = 9 a result within tolerance fails one row test with
#     probability below 5e-18, below 1e-12 over all rows and vectors of a
#     16384^3 check. It catches far smaller errors than the summed bound:
#     wrong or missing tiles, rows, columns, scale blocks, K blocks.
# Both also allow the double rounding of y (gamma_{K+1} g) and of z
# (gamma_N sum_j |D_ij|), and BF16's subnormal spacing (2^-133 per term).

FREIVALDS_C = 9.0
_U = 2.0 ** -53
_RHO = REL_TOL + 2.0 ** -8 / (1.0 - 2.0 ** -8)
_C1 = _RHO / (1.0 - REL_TOL)
_C2 = ABS_TOL * (1.0 + _C1)


def rademacher(nv: int, n: int, seed: int) -> np.ndarray:
    """nv vectors of n independent +-1 entries (int8), seeded (PCG64)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return (rng.integers(0, 2, size=(nv, n), dtype=np.int8) * 2 - 1).astype(np.int8)


def bf16_times_vectors(d_bits, x, chunk_rows: int = 1024):
    """z = D x in double for BF16 D (uint16 bits [M, N]) and x [nv, N], and
    the row sums the bounds need: returns (z [nv, M], abs_sum [M] =
    sum_j |D_ij|, sq_sum [M] = sum_j D_ij^2, nonfinite [M] = count of Inf /
    NaN in the row, which are left out of the other three). Chunked over rows."""
    d_bits = np.asarray(d_bits, dtype=np.uint16)
    M, N = d_bits.shape
    xv = np.asarray(x, dtype=np.float64)
    assert xv.shape[1] == N
    z = np.empty((xv.shape[0], M))
    abs_sum = np.empty(M)
    sq_sum = np.empty(M)
    nonfinite = np.empty(M, np.int64)
    for r0 in range(0, M, chunk_rows):
        d = bf16_bits_to_float(d_bits[r0:r0 + chunk_rows])
        bad = ~np.isfinite(d)
        nonfinite[r0:r0 + d.shape[0]] = bad.sum(axis=1)
        d[bad] = 0.0
        z[:, r0:r0 + d.shape[0]] = (d @ xv.T).T
        a = np.abs(d)
        abs_sum[r0:r0 + d.shape[0]] = a.sum(axis=1)
        sq_sum[r0:r0 + d.shape[0]] = (a * a).sum(axis=1)
    return z, abs_sum, sq_sum, nonfinite


def freivalds_outcome(d_bits, x, rhs) -> dict:
    """Decide Freivalds' check of the GPU result d_bits (BF16 bits [M, N])
    against the oracle's right-hand side rhs (from nvfp4_freivalds /
    fp8_freivalds with the same x). Returns a dict with 'ok' (both bounds
    hold everywhere and every element is finite), 'ok_summed', 'ok_hoeffding',
    the worst ratios |r| / bound of each, and the failing (vector, row) pairs
    of the Hoeffding bound (up to 16)."""
    x = np.asarray(x, dtype=np.int8)
    M, N = np.asarray(d_bits).shape
    if not np.all(np.abs(x.astype(np.int16)) == 1):
        raise ValueError("Freivalds vectors must hold +-1 entries only")
    z, abs_sum, sq_sum, nonfinite = bf16_times_vectors(d_bits, x)
    y, g, tsum, t2, K = rhs["y"], rhs["g"], rhs["tsum"], rhs["t2"], rhs["K"]
    gam_n = N * _U / (1.0 - N * _U)
    gam_k = (K + 2) * _U / (1.0 - (K + 2) * _U)
    r = np.abs(z - y)
    rounding = gam_n * abs_sum[None, :] + gam_k * g + N * 2.0 ** -133
    summed = _C1 * abs_sum + _C2 * tsum * (1.0 + gam_k)
    summed = summed[None, :] + rounding
    sigma = _C1 * np.sqrt(sq_sum) + _C2 * np.sqrt(t2 * (1.0 + gam_k))
    hoeff = FREIVALDS_C * sigma[None, :] + rounding
    with np.errstate(invalid="ignore", divide="ignore"):
        ratio_s = np.where(summed > 0, r / summed, np.where(r > 0, np.inf, 0.0))
        ratio_h = np.where(hoeff > 0, r / hoeff, np.where(r > 0, np.inf, 0.0))
    ok_s = bool((ratio_s <= 1.0).all())
    ok_h = bool((ratio_h <= 1.0).all())
    finite = bool((nonfinite == 0).all())
    fails = np.argwhere(~(ratio_h <= 1.0))[:16]
    return dict(ok=ok_s and ok_h and finite, ok_summed=ok_s, ok_hoeffding=ok_h, finite=finite,
                worst_summed=float(np.nanmax(ratio_s)), worst_hoeffding=float(np.nanmax(ratio_h)),
                fails=[(int(q), int(i)) for q, i in fails])
