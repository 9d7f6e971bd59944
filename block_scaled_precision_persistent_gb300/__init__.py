"""Block-scaled NVFP4 / FP8 GEMM for one GB300 GPU (sm_103a).

    D = alpha * (A (.) sA)(B (.) sB)^T      FP32 accumulation, BF16 output

Thin Python binding of the C ABI in ``include/bsgemm.h`` (``libbsgemm.so``,
built in-tree by ``_build.build()``). Every function here has the name of its
C entry point and only marshals arguments: tensors become device pointers,
``stream=None`` becomes PyTorch's current CUDA stream, and a non-zero status
raises :class:`BsgError`. All arithmetic runs in the library's CUDA kernels;
there is no fallback. If the library is missing, the first call raises.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

__all__ = [
    "BsgError", "load", "nvfp4_gemm", "nvfp4_gemm_swizzled", "nvfp4_swizzle_scales", "nvfp4_quantize",
    "nvfp4_swizzled_scale_bytes", "nvfp4_gemm_noalloc", "fp8_gemm", "nvfp4_gemm_ex", "fp8_gemm_ex",
    "nvfp4_grouped_gemm", "nvfp4_swizzle_scales_grouped", "nvfp4_grouped_scale_bytes", "nvfp4_dense_gemm",
    "nvfp4_dense_f16_gemm", "nvfp4_dense_grouped_gemm", "nvfp4_dense_f16_grouped_gemm",
    "nvfp4_dense_kgrouped_gemm", "nvfp4_dense_f16_kgrouped_gemm",
    "nvfp4_swizzle_scales2", "nvfp4_quantize_tiles", "nvfp4_pack_operand", "nvfp4_packed_operand_bytes", "nvfp4_gemm_packed", "nvfp4_gemm_packed_ex",
    "bsg_reserve_workspace", "bsg_get_device_status",
    "bsg_last_status_word", "bsg_set_watchdog_ns", "bsg_set_raster_group", "bsg_set_skinny_splits", "bsg_set_pdl", "bsg_watchdog_selftest", "bsg_force_plan",
    "bsg_measure_ingress",
    "bsg_select_plan", "bsg_last_launch_count", "bsg_last_plan_name", "bsg_error_string", "EXPORTED_SYMBOLS",
    "BSG_OK", "BSG_ERR_INVALID_ARG", "BSG_ERR_MISALIGNED", "BSG_ERR_UNSUPPORTED_DEVICE",
    "BSG_ERR_NO_PLAN", "BSG_ERR_CUDA", "BSG_ERR_DEVICE_TIMEOUT", "BSG_ERR_OUT_OF_MEMORY",
    "BSG_ERR_EXCEEDS_SCRATCH", "BSG_NOALLOC_SCRATCH_BYTES",
]

BSG_OK = 0
BSG_ERR_INVALID_ARG = 1
BSG_ERR_MISALIGNED = 2
BSG_ERR_UNSUPPORTED_DEVICE = 3
BSG_ERR_NO_PLAN = 4
BSG_ERR_CUDA = 5
BSG_ERR_DEVICE_TIMEOUT = 6
BSG_ERR_OUT_OF_MEMORY = 7
BSG_ERR_EXCEEDS_SCRATCH = 8
BSG_NOALLOC_SCRATCH_BYTES = 16 << 20     # fixed scratch of nvfp4_gemm_noalloc

LIB_PATH = Path(__file__).resolve().parent / "libbsgemm.so"

_vp = ctypes.c_void_p
_i = ctypes.c_int
# name -> (restype, argtypes), in the order of include/bsgemm.h
_SIGNATURES = {
    "nvfp4_gemm": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "nvfp4_gemm_swizzled": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "nvfp4_packed_operand_bytes": (ctypes.c_size_t, [_i, _i]),
    "nvfp4_pack_operand": (_i, [_i, _i, _vp, _vp, _vp]),
    "nvfp4_gemm_packed": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "nvfp4_gemm_packed_ex": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp, _vp]),
    "nvfp4_swizzle_scales": (_i, [_i, _i, _vp, _vp, _vp]),
    "nvfp4_swizzle_scales2": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_swizzled_scale_bytes": (ctypes.c_size_t, [_i, _i]),
    "nvfp4_quantize": (_i, [_i, _i, _vp, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_quantize_tiles": (_i, [_i, _i, _vp, _vp, _vp, _vp, _vp, _vp]),
    "nvfp4_gemm_noalloc": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "fp8_gemm": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp]),
    "nvfp4_gemm_ex": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp, _vp]),
    "fp8_gemm_ex": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp, _vp]),
    "nvfp4_dense_gemm": (_i, [_i, _i, _i, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp, _vp]),
    "nvfp4_dense_f16_gemm": (_i, [_i, _i, _i, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp, _vp]),
    "nvfp4_dense_grouped_gemm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp,
                                      _vp]),
    "nvfp4_dense_kgrouped_gemm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]),
    "nvfp4_dense_f16_kgrouped_gemm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp,
                                           _vp]),
    "nvfp4_dense_f16_grouped_gemm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i,
                                          _vp, _vp]),
    "nvfp4_grouped_gemm": (_i, [_i, _i, _i, _i, _vp, _vp, _vp, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _i, _vp,
                                _vp]),
    "nvfp4_swizzle_scales_grouped": (_i, [_i, _i, _i, _vp, _vp, _vp, _vp]),
    "nvfp4_grouped_scale_bytes": (ctypes.c_size_t, [_i, _i, _i]),
    "bsg_reserve_workspace": (_i, [_i, ctypes.c_size_t]),
    "bsg_get_device_status": (_i, [_vp]),
    "bsg_last_status_word": (ctypes.c_uint32, []),
    "bsg_set_watchdog_ns": (_i, [ctypes.c_uint64]),
    "bsg_set_raster_group": (_i, [_i]),
    "bsg_set_skinny_splits": (_i, [_i]),
    "bsg_set_pdl": (_i, [_i]),
    "bsg_watchdog_selftest": (_i, [ctypes.c_uint64, _vp]),
    "bsg_measure_ingress": (_i, [ctypes.c_size_t, _i, _i, ctypes.POINTER(ctypes.c_double),
                                 ctypes.POINTER(ctypes.c_double)]),
    "bsg_force_plan": (_i, [ctypes.c_char_p]),
    "bsg_select_plan": (_i, [_i, _i, _i, _i, _i, ctypes.c_char_p, ctypes.c_size_t]),
    "bsg_last_launch_count": (_i, []),
    "bsg_last_plan_name": (ctypes.c_char_p, []),
    "bsg_error_string": (ctypes.c_char_p, [_i]),
}
EXPORTED_SYMBOLS = tuple(_SIGNATURES)

_lib: ctypes.CDLL | None = None


class BsgError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {bsg_error_string(code)} (status {code})")


def load() -> ctypes.CDLL:
    """Load libbsgemm.so (built in-tree). Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not LIB_PATH.exists():
            raise ImportError(f"{LIB_PATH.name} is not built; run __graft_entry__.build() "
                              "(or python -m block_scaled_precision_persistent_gb300._build)")
        lib = ctypes.CDLL(str(LIB_PATH))
        for name, (res, args) in _SIGNATURES.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
    return _lib


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(s) -> int | None:
    if s is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream) if torch.cuda.is_available() else None
    if isinstance(s, int):
        return s
    return int(s.cuda_stream)


def _check(rc: int, where: str) -> None:
    if rc != BSG_OK:
        raise BsgError(rc, where)


def nvfp4_gemm(M, N, K, A, sfA, B, sfB, alpha, D, stream=None) -> None:
    """D[M,N] bf16 = alpha * (A*sA)(B*sB)^T with row-major uint8[rows, K/16] scales."""
    _check(load().nvfp4_gemm(M, N, K, _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB), float(alpha),
                             _ptr(D), _stream(stream)), "nvfp4_gemm")


def nvfp4_gemm_swizzled(M, N, K, A, sfA_swz, B, sfB_swz, alpha, D, stream=None) -> None:
    """As nvfp4_gemm, with scales already in the swizzled layout."""
    _check(load().nvfp4_gemm_swizzled(M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(sfB_swz),
                                      float(alpha), _ptr(D), _stream(stream)), "nvfp4_gemm_swizzled")


def nvfp4_packed_operand_bytes(rows, K) -> int:
    """Bytes of an operand of `rows` rows in the tile-packed layout (0 if invalid)."""
    return int(load().nvfp4_packed_operand_bytes(rows, K))


def nvfp4_pack_operand(rows, K, X, out, stream=None) -> None:
    """uint8[rows, K/2] NVFP4 codes -> the tile-packed layout (16 KiB tiles
    of 128 rows x 128 bytes, 128-byte swizzled inside, rows padded with zeros)."""
    _check(load().nvfp4_pack_operand(rows, K, _ptr(X), _ptr(out), _stream(stream)), "nvfp4_pack_operand")


def nvfp4_gemm_packed(M, N, K, A_packed, sfA_swz, B_packed, sfB_swz, alpha, D, stream=None) -> None:
    """As nvfp4_gemm_swizzled, with A and B in the tile-packed layout."""
    _check(load().nvfp4_gemm_packed(M, N, K, _ptr(A_packed), _ptr(sfA_swz), _ptr(B_packed), _ptr(sfB_swz),
                                    float(alpha), _ptr(D), _stream(stream)), "nvfp4_gemm_packed")


def nvfp4_gemm_packed_ex(M, N, K, A_packed, sfA_swz, B_packed, sfB_swz, alpha, bias, gamma, scatter, m_out, D,
                         stream=None) -> None:
    """As nvfp4_gemm_packed, with the epilogue variants of nvfp4_gemm_ex."""
    _check(load().nvfp4_gemm_packed_ex(M, N, K, _ptr(A_packed), _ptr(sfA_swz), _ptr(B_packed), _ptr(sfB_swz),
                                       float(alpha), _ptr(bias), _ptr(gamma), _ptr(scatter), int(m_out), _ptr(D),
                                       _stream(stream)), "nvfp4_gemm_packed_ex")


def nvfp4_swizzle_scales(rows, K, sf, sf_swz, stream=None) -> None:
    _check(load().nvfp4_swizzle_scales(rows, K, _ptr(sf), _ptr(sf_swz), _stream(stream)),
           "nvfp4_swizzle_scales")


def nvfp4_swizzle_scales2(M, N, K, sfA, sfA_swz, sfB, sfB_swz, stream=None) -> None:
    """Both operands' scales of one GEMM into the swizzled layout, one launch."""
    _check(load().nvfp4_swizzle_scales2(M, N, K, _ptr(sfA), _ptr(sfA_swz), _ptr(sfB), _ptr(sfB_swz),
                                        _stream(stream)), "nvfp4_swizzle_scales2")


def nvfp4_swizzled_scale_bytes(rows, K) -> int:
    return int(load().nvfp4_swizzled_scale_bytes(rows, K))


def nvfp4_quantize_tiles(rows, K, X, packed_tiles, sf_swz, sf_rowmajor, global_scales, stream=None) -> None:
    """As nvfp4_quantize, with the codes written in the tile-packed layout
    nvfp4_gemm_packed reads (K % 256 == 0)."""
    _check(load().nvfp4_quantize_tiles(rows, K, _ptr(X), _ptr(packed_tiles), _ptr(sf_swz), _ptr(sf_rowmajor),
                                       _ptr(global_scales), _stream(stream)), "nvfp4_quantize_tiles")


def nvfp4_quantize(rows, K, X, packed, sf_swz, sf_rowmajor, global_scales, stream=None) -> None:
    """Two-level NVFP4 quantisation of BF16 X[rows, K] into packed codes,
    swizzled (and optionally row-major) E4M3 block scales, and
    global_scales[0:2] = (amax, s_g) on the device; alpha for the GEMM is
    1 / (s_gA * s_gB)."""
    _check(load().nvfp4_quantize(rows, K, _ptr(X), _ptr(packed), _ptr(sf_swz), _ptr(sf_rowmajor),
                                 _ptr(global_scales), _stream(stream)), "nvfp4_quantize")


def nvfp4_gemm_noalloc(M, N, K, A, sfA, B, sfB, alpha, D, stream=None) -> None:
    """As nvfp4_gemm, but the swizzled scales go to the library's fixed device
    scratch array (BSG_NOALLOC_SCRATCH_BYTES) instead of an allocated
    workspace: for callers that cannot allocate device memory. Calls whose
    work overlaps on the GPU share that array and race."""
    _check(load().nvfp4_gemm_noalloc(M, N, K, _ptr(A), _ptr(sfA), _ptr(B), _ptr(sfB),
                                     float(alpha), _ptr(D), _stream(stream)), "nvfp4_gemm_noalloc")


def fp8_gemm(M, N, K, A, sA, B, sB, alpha, D, stream=None) -> None:
    """D = alpha*sA*sB * A B^T, E4M3 operands; sA/sB device float tensors or None."""
    _check(load().fp8_gemm(M, N, K, _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), float(alpha), _ptr(D),
                           _stream(stream)), "fp8_gemm")


def nvfp4_gemm_ex(M, N, K, A, sfA_swz, B, sfB_swz, alpha, bias, gamma, scatter, m_out, D,
                  stream=None) -> None:
    """As nvfp4_gemm_swizzled with the fused epilogue
    D[scatter[m]][n] = bf16(gamma[m] * (alpha * acc[m][n] + bias[n])):
    bias float32[N], gamma float32[M], scatter int32[M] (each None to omit);
    D has m_out rows (m_out == M without scatter)."""
    _check(load().nvfp4_gemm_ex(M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(sfB_swz), float(alpha),
                                _ptr(bias), _ptr(gamma), _ptr(scatter), int(m_out), _ptr(D),
                                _stream(stream)), "nvfp4_gemm_ex")


def fp8_gemm_ex(M, N, K, A, sA, B, sB, alpha, bias, gamma, scatter, m_out, D, stream=None) -> None:
    """As fp8_gemm with the fused epilogue of nvfp4_gemm_ex."""
    _check(load().fp8_gemm_ex(M, N, K, _ptr(A), _ptr(sA), _ptr(B), _ptr(sB), float(alpha), _ptr(bias),
                              _ptr(gamma), _ptr(scatter), int(m_out), _ptr(D), _stream(stream)),
           "fp8_gemm_ex")


def nvfp4_dense_gemm(M, N, K, A, sfA_swz, B, alpha, bias, gamma, scatter, m_out, D, stream=None) -> None:
    """NVFP4 activations (E2M1 codes + swizzled E4M3 scales) times dense BF16
    weights B[N, K]; the epilogue as nvfp4_gemm_ex."""
    _check(load().nvfp4_dense_gemm(M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), float(alpha), _ptr(bias), _ptr(gamma),
                                   _ptr(scatter), int(m_out), _ptr(D), _stream(stream)), "nvfp4_dense_gemm")


def nvfp4_dense_f16_gemm(M, N, K, A, sfA_swz, B, alpha, bias, gamma, scatter, m_out, D, stream=None) -> None:
    """As nvfp4_dense_gemm with FP16 weights B[N, K]."""
    _check(load().nvfp4_dense_f16_gemm(M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), float(alpha), _ptr(bias),
                                       _ptr(gamma), _ptr(scatter), int(m_out), _ptr(D), _stream(stream)),
           "nvfp4_dense_f16_gemm")


def nvfp4_grouped_gemm(E, M, N, K, A, sfA_swz, B, sfB_swz, offs, alpha, bias, gamma, scatter, m_out, D,
                       stream=None) -> None:
    """Grouped (ragged, routed) NVFP4 GEMM: rows [offs[e], offs[e+1]) of A
    times B[e]^T for each of the E slices; offs is a device int32[E+1]
    tensor, B uint8[E, N, K/2], bias float32[E, N] or None; the epilogue as
    nvfp4_gemm_ex."""
    _check(load().nvfp4_grouped_gemm(E, M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(sfB_swz), _ptr(offs),
                                     float(alpha), _ptr(bias), _ptr(gamma), _ptr(scatter), int(m_out), _ptr(D),
                                     _stream(stream)), "nvfp4_grouped_gemm")


def nvfp4_swizzle_scales_grouped(E, M, K, offs, sf, sf_swz, stream=None) -> None:
    """Per-slice scale layout of a grouped A (see nvfp4_grouped_gemm)."""
    _check(load().nvfp4_swizzle_scales_grouped(E, M, K, _ptr(offs), _ptr(sf), _ptr(sf_swz), _stream(stream)),
           "nvfp4_swizzle_scales_grouped")


def nvfp4_grouped_scale_bytes(E, M, K) -> int:
    return int(load().nvfp4_grouped_scale_bytes(E, M, K))


def bsg_reserve_workspace(device: int, nbytes: int) -> None:
    _check(load().bsg_reserve_workspace(device, nbytes), "bsg_reserve_workspace")


def bsg_get_device_status(stream=None) -> int:
    """Synchronise and return (and clear) the device status code; does not raise."""
    return int(load().bsg_get_device_status(_stream(stream)))


def bsg_last_status_word() -> int:
    return int(load().bsg_last_status_word())


def bsg_set_watchdog_ns(ns: int) -> None:
    _check(load().bsg_set_watchdog_ns(ns), "bsg_set_watchdog_ns")


def bsg_set_pdl(on: "bool | int") -> None:
    """Programmatic dependent launch for later GEMM launches (off by default):
    False/0 off, True/1 on, 2 on with B's codes read before the wait for the
    previous kernel (the caller promises that kernel does not write them)."""
    _check(load().bsg_set_pdl(int(on)), "bsg_set_pdl")


def bsg_set_raster_group(m_tiles: int) -> None:
    """M tiles per rasterisation group for later launches (0: default 16)."""
    _check(load().bsg_set_raster_group(int(m_tiles)), "bsg_set_raster_group")


def bsg_set_skinny_splits(splits: int) -> None:
    """K splits of the skinny-M kernel for later launches (0: chosen per call)."""
    _check(load().bsg_set_skinny_splits(int(splits)), "bsg_set_skinny_splits")


def bsg_watchdog_selftest(ns: int, stream=None) -> None:
    _check(load().bsg_watchdog_selftest(ns, _stream(stream)), "bsg_watchdog_selftest")


def nvfp4_dense_grouped_gemm(E, M, N, K, A, sfA_swz, B, offs, alpha, bias, gamma, scatter, m_out, D,
                             stream=None) -> None:
    """Grouped (routed) NVFP4 x dense BF16 GEMM: rows offs[e]..offs[e+1] of A
    times B[e] (bf16 [E, N, K]); the epilogue as nvfp4_grouped_gemm."""
    _check(load().nvfp4_dense_grouped_gemm(E, M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(offs), float(alpha),
                                           _ptr(bias), _ptr(gamma), _ptr(scatter), int(m_out), _ptr(D),
                                           _stream(stream)), "nvfp4_dense_grouped_gemm")


def nvfp4_dense_f16_grouped_gemm(E, M, N, K, A, sfA_swz, B, offs, alpha, bias, gamma, scatter, m_out, D,
                                 stream=None) -> None:
    """As nvfp4_dense_grouped_gemm with FP16 right-hand sides."""
    _check(load().nvfp4_dense_f16_grouped_gemm(E, M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(offs),
                                               float(alpha), _ptr(bias), _ptr(gamma), _ptr(scatter), int(m_out),
                                               _ptr(D), _stream(stream)), "nvfp4_dense_f16_grouped_gemm")


def nvfp4_dense_kgrouped_gemm(E, M, N, K, A, sfA_swz, B, koffs, alpha, bias, gamma, D, stream=None) -> None:
    """Inner-expert (K-ragged) NVFP4 x dense BF16 GEMM: slice e of K (koffs,
    device int32[E+1]) gives D[e] (bf16 [E, M, N]) with bias[e] and gamma."""
    _check(load().nvfp4_dense_kgrouped_gemm(E, M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(koffs), float(alpha),
                                            _ptr(bias), _ptr(gamma), _ptr(D), _stream(stream)),
           "nvfp4_dense_kgrouped_gemm")


def nvfp4_dense_f16_kgrouped_gemm(E, M, N, K, A, sfA_swz, B, koffs, alpha, bias, gamma, D, stream=None) -> None:
    """As nvfp4_dense_kgrouped_gemm with an FP16 right-hand side."""
    _check(load().nvfp4_dense_f16_kgrouped_gemm(E, M, N, K, _ptr(A), _ptr(sfA_swz), _ptr(B), _ptr(koffs),
                                                float(alpha), _ptr(bias), _ptr(gamma), _ptr(D), _stream(stream)),
           "nvfp4_dense_f16_kgrouped_gemm")


def bsg_measure_ingress(src_bytes: int = 32 << 20, stages: int = 4, tensor_boxes: bool = False) -> tuple[float, float]:
    """Operand-ingress probe: (bytes per SM clock cycle per SM, total GB/s);
    contiguous bulk copies, or tensor-map boxes of 128 rows x 128 bytes."""
    per_sm, total = ctypes.c_double(0.0), ctypes.c_double(0.0)
    _check(load().bsg_measure_ingress(int(src_bytes), int(stages), 1 if tensor_boxes else 0, ctypes.byref(per_sm),
                                      ctypes.byref(total)), "bsg_measure_ingress")
    return per_sm.value, total.value


def bsg_force_plan(name: str | None) -> None:
    _check(load().bsg_force_plan(name.encode() if name else None), "bsg_force_plan")


def bsg_select_plan(kind: int, M: int, N: int, K: int, num_sms: int) -> str:
    buf = ctypes.create_string_buffer(128)
    _check(load().bsg_select_plan(kind, M, N, K, num_sms, buf, len(buf)), "bsg_select_plan")
    return buf.value.decode()


def bsg_last_launch_count() -> int:
    return int(load().bsg_last_launch_count())


def bsg_last_plan_name() -> str:
    """Plan of the last GEMM launch on this thread ("" before any)."""
    return load().bsg_last_plan_name().decode()


def bsg_error_string(code: int) -> str:
    try:
        return load().bsg_error_string(code).decode()
    except ImportError:
        return f"status {code}"
