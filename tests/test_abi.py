"""Host-side checks of the C ABI (no GPU): the library loads, exports every
entry point the header declares, rejects bad arguments before launching
anything, and its planner and error strings behave."""
import re
from pathlib import Path

import pytest

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg

ROOT = Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return bsg.load()


def header_functions():
    text = (ROOT / "include" / "bsgemm.h").read_text()
    return re.findall(r"^BSG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text, re.M)


def test_header_and_binding_agree():
    names = header_functions()
    assert len(names) >= 14
    assert sorted(names) == sorted(bsg.EXPORTED_SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in header_functions():
        assert hasattr(lib, name), name


def test_only_declared_symbols_are_exported(lib):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", str(bsg.LIB_PATH)], capture_output=True,
                         text=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    ours = {n for n in exported if not n.startswith("_")}
    assert ours == set(header_functions()), ours ^ set(header_functions())


BAD = 0x1000  # a non-null, 16-byte-aligned fake pointer: never dereferenced


@pytest.mark.parametrize("M,N,K", [(0, 8, 256), (8, 0, 256), (8, 8, 128), (8, 8, 300), (8, 12, 256),
                                   (-1, 8, 256)])
def test_nvfp4_bad_sizes(lib, M, N, K):
    for fn in (lib.nvfp4_gemm, lib.nvfp4_gemm_swizzled):
        assert fn(M, N, K, BAD, BAD, BAD, BAD, 1.0, BAD, None) == bsg.BSG_ERR_INVALID_ARG


def test_nvfp4_null_and_misaligned(lib):
    assert lib.nvfp4_gemm(128, 128, 256, None, BAD, BAD, BAD, 1.0, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.nvfp4_gemm(128, 128, 256, BAD + 8, BAD, BAD, BAD, 1.0, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert lib.nvfp4_gemm_swizzled(128, 128, 256, BAD, BAD, BAD, BAD, 1.0, BAD + 2, None) == \
        bsg.BSG_ERR_MISALIGNED


def test_fp8_bad_args(lib):
    assert lib.fp8_gemm(128, 128, 64, BAD, None, BAD, None, 1.0, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.fp8_gemm(128, 128, 128, None, None, BAD, None, 1.0, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.fp8_gemm(128, 128, 128, BAD, BAD + 1, BAD, None, 1.0, BAD, None) == bsg.BSG_ERR_MISALIGNED


def test_swizzle_bad_args(lib):
    assert lib.nvfp4_swizzle_scales(0, 256, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.nvfp4_swizzle_scales(8, 24, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.nvfp4_swizzle_scales(8, 256, BAD, BAD + 4, None) == bsg.BSG_ERR_MISALIGNED
    s2 = lib.nvfp4_swizzle_scales2
    assert s2(0, 8, 256, BAD, BAD, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s2(8, 0, 256, BAD, BAD, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s2(8, 8, 24, BAD, BAD, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s2(8, 8, 256, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s2(8, 8, 256, BAD, BAD + 4, BAD, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert s2(8, 8, 256, BAD, BAD, BAD, BAD + 8, None) == bsg.BSG_ERR_MISALIGNED


def test_swizzled_bytes(lib):
    assert bsg.nvfp4_swizzled_scale_bytes(1, 16) == 128 * 4
    assert bsg.nvfp4_swizzled_scale_bytes(128, 256) == 128 * 16
    assert bsg.nvfp4_swizzled_scale_bytes(300, 1040) == 384 * 68
    assert bsg.nvfp4_swizzled_scale_bytes(16384, 16384) == 16384 * 1024
    assert bsg.nvfp4_swizzled_scale_bytes(10, 24) == 0


def test_planner_enumeration(lib):
    # every shape picks a plan of its own kind, by the planner's rules
    sms = 152
    for kind, prefix in ((0, "nvfp4_"), (1, "fp8_")):
        for M in (1, 64, 65, 128, 129, 256, 257, 512, 4096, 16384):
            for N in (8, 128, 136, 256, 3072, 12288, 16384):
                for K in (256, 4096, 12288):
                    name = bsg.bsg_select_plan(kind, M, N, K, sms)
                    assert name.startswith(prefix), name
                    tiles128 = -(-M // 128) * -(-N // 128)
                    few = tiles128 <= 4 * sms
                    if kind == 1:
                        assert ("x128_" in name) == (N <= 128), (N, name)
                        assert ("_tc2_" in name) == (M > 128 and N > 128), (M, N, name)
                        continue
                    split = 2 * -(-N // 128) <= sms and K >= 512
                    pair_tiles = -(-M // 256) * -(-N // 256)
                    if split and (M <= 64 or (M <= 256 and K >= 8192)):
                        mpad = 64 if M <= 64 else 128 if M <= 128 else 256
                        assert name.startswith(f"nvfp4_skinny_m{mpad}_"), (M, N, K, name)
                    elif 128 < M <= 512 and N > 128 and 4 * pair_tiles >= sms:
                        assert name == "nvfp4_tc2_256x256_s5_acc1", (M, N, K, name)
                    elif few or N <= 128:
                        want = "tc1_128x128" if (M <= 128 or few) else "tc2_256x128"
                        assert want in name, (M, N, K, name)
                    else:
                        want = "tc1_128x256" if M <= 128 else "tc2_256x256"
                        assert want in name, (M, N, K, name)


def test_planner_headline_shapes(lib):
    # the shapes the benchmarks time
    assert bsg.bsg_select_plan(0, 16384, 16384, 16384, 152) == "nvfp4_tc2_256x256_s5_acc1"
    assert bsg.bsg_select_plan(1, 8192, 8192, 8192, 152) == "fp8_tc2_256x512_s4_acc1"
    assert bsg.bsg_select_plan(1, 8192, 8448, 8192, 152) == "fp8_tc2_256x256_s6_acc2"   # N not whole 512s
    assert bsg.bsg_select_plan(1, 128, 8192, 8192, 152) == "fp8_tc1_128x256_s4_acc2"
    assert bsg.bsg_select_plan(0, 64, 3072, 3072, 152) == "nvfp4_skinny_m64_s3"
    assert bsg.bsg_select_plan(0, 64, 3072, 12288, 152) == "nvfp4_skinny_m64_s6"
    assert bsg.bsg_select_plan(0, 256, 3072, 12288, 152) == "nvfp4_skinny_m256_s4"
    assert bsg.bsg_select_plan(0, 256, 3072, 3072, 152) == "nvfp4_tc1_128x128_s5_acc2"
    assert bsg.bsg_select_plan(0, 128, 3072, 3072, 152) == "nvfp4_tc1_128x128_s5_acc2"
    assert bsg.bsg_select_plan(0, 256, 12288, 3072, 152) == "nvfp4_tc2_256x256_s5_acc1"
    assert bsg.bsg_select_plan(0, 512, 12288, 3072, 152) == "nvfp4_tc2_256x256_s5_acc1"
    assert bsg.bsg_select_plan(0, 512, 3072, 12288, 152) == "nvfp4_tc1_128x128_s5_acc2"


def test_forced_skinny_plan_needs_small_m(lib):
    bsg.bsg_force_plan("nvfp4_skinny_m64_s6")
    try:
        assert bsg.bsg_select_plan(0, 64, 3072, 3072, 152) == "nvfp4_skinny_m64_s6"
        with pytest.raises(bsg.BsgError):       # 65 activation rows do not fit
            bsg.bsg_select_plan(0, 65, 3072, 3072, 152)
    finally:
        bsg.bsg_force_plan(None)
    bsg.bsg_force_plan("nvfp4_skinny_m256_s4")   # two blocks of 256 activation rows
    try:
        assert bsg.bsg_select_plan(0, 512, 3072, 3072, 152) == "nvfp4_skinny_m256_s4"
        with pytest.raises(bsg.BsgError):
            bsg.bsg_select_plan(0, 513, 3072, 3072, 152)
    finally:
        bsg.bsg_force_plan(None)


def test_skinny_splits_lever(lib):
    for bad in (-1, 7, 9):
        with pytest.raises(bsg.BsgError) as e:
            bsg.bsg_set_skinny_splits(bad)
        assert e.value.code == bsg.BSG_ERR_INVALID_ARG
    for good in (1, 2, 3, 4, 5, 6, 8, 0):
        bsg.bsg_set_skinny_splits(good)


def test_pdl_lever(lib):
    for bad in (-1, 3):
        assert lib.bsg_set_pdl(bad) == bsg.BSG_ERR_INVALID_ARG
    for good in (2, True, 1, False):
        bsg.bsg_set_pdl(good)
    bsg.bsg_set_pdl(False)


def test_forced_plan(lib):
    with pytest.raises(bsg.BsgError) as e:
        bsg.bsg_force_plan("no_such_plan")
    assert e.value.code == bsg.BSG_ERR_NO_PLAN
    bsg.bsg_force_plan("nvfp4_tc1_128x128_s5_acc2")
    try:
        assert bsg.bsg_select_plan(0, 4096, 4096, 4096, 152) == "nvfp4_tc1_128x128_s5_acc2"
        with pytest.raises(bsg.BsgError):       # an NVFP4 plan cannot serve FP8
            bsg.bsg_select_plan(1, 4096, 4096, 4096, 152)
    finally:
        bsg.bsg_force_plan(None)
    assert bsg.bsg_select_plan(0, 4096, 4096, 4096, 152) == "nvfp4_tc2_256x256_s5_acc1"


def test_error_strings(lib):
    assert bsg.bsg_error_string(0) == "ok"
    assert "timed out" in bsg.bsg_error_string(bsg.BSG_ERR_DEVICE_TIMEOUT)
    assert bsg.bsg_error_string(99) == "unknown status"


def test_quantize_bad_args(lib):
    q = lib.nvfp4_quantize
    assert q(0, 256, BAD, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert q(8, 24, BAD, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG          # K % 16
    assert q(8, 256, None, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert q(8, 256, BAD, BAD, BAD, None, None, None) == bsg.BSG_ERR_INVALID_ARG         # no global
    assert q(8, 256, BAD + 2, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_MISALIGNED       # X
    assert q(8, 256, BAD, BAD + 8, BAD, None, BAD, None) == bsg.BSG_ERR_MISALIGNED       # packed
    assert q(8, 256, BAD, BAD, BAD + 4, None, BAD, None) == bsg.BSG_ERR_MISALIGNED       # sf_swz
    assert q(8, 256, BAD, BAD, BAD, None, BAD + 4, None) == bsg.BSG_ERR_MISALIGNED       # global
    t = lib.nvfp4_quantize_tiles
    assert t(8, 48, BAD, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG          # K % 256
    assert t(8, 768 + 16, BAD, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert t(0, 256, BAD, BAD, BAD, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert t(8, 256, BAD, BAD + 8, BAD, None, BAD, None) == bsg.BSG_ERR_MISALIGNED       # tiles


def test_epilogue_bad_args(lib):
    """nvfp4_gemm_ex / fp8_gemm_ex: operand checks as the plain calls, then
    m_out == M without scatter (>= 1 with it), bias 16-byte and gamma /
    scatter 4-byte alignment; all rejected before any launch."""
    nv = lambda *e: lib.nvfp4_gemm_ex(128, 64, 256, BAD, BAD, BAD, BAD, 1.0, *e, BAD, None)  # noqa: E731
    f8 = lambda *e: lib.fp8_gemm_ex(128, 64, 128, BAD, None, BAD, None, 1.0, *e, BAD, None)  # noqa: E731
    for fn in (nv, f8):
        assert fn(None, None, None, 100) == bsg.BSG_ERR_INVALID_ARG            # m_out != M
        assert fn(BAD, None, None, 127) == bsg.BSG_ERR_INVALID_ARG
        assert fn(None, None, BAD, 0) == bsg.BSG_ERR_INVALID_ARG               # scatter, no rows
        assert fn(BAD + 4, None, None, 128) == bsg.BSG_ERR_MISALIGNED          # bias
        assert fn(None, BAD + 2, None, 128) == bsg.BSG_ERR_MISALIGNED          # gamma
        assert fn(None, None, BAD + 1, 7) == bsg.BSG_ERR_MISALIGNED            # scatter
    assert lib.nvfp4_gemm_ex(128, 64, 300, BAD, BAD, BAD, BAD, 1.0, None, None, None, 128, BAD, None) == \
        bsg.BSG_ERR_INVALID_ARG
    assert lib.fp8_gemm_ex(128, 64, 128, BAD, BAD + 1, BAD, None, 1.0, None, None, None, 128, BAD, None) == \
        bsg.BSG_ERR_MISALIGNED
    assert lib.nvfp4_gemm_ex(128, 64, 256, BAD, BAD, BAD, BAD, 1.0, None, None, None, 128, None, None) == \
        bsg.BSG_ERR_INVALID_ARG                                                # no D


def test_grouped_bad_args(lib):
    """nvfp4_grouped_gemm / nvfp4_swizzle_scales_grouped reject bad slice
    counts, missing offsets and misalignment before any launch."""
    g = lambda E, offs, *rest: lib.nvfp4_grouped_gemm(E, 128, 64, 256, BAD, BAD, BAD, BAD, offs, 1.0,  # noqa: E731
                                                      *rest)
    ok_epi = (None, None, None, 128, BAD, None)
    assert g(0, BAD, *ok_epi) == bsg.BSG_ERR_INVALID_ARG                     # no slices
    assert g(1025, BAD, *ok_epi) == bsg.BSG_ERR_INVALID_ARG                  # too many slices
    assert g(4, None, *ok_epi) == bsg.BSG_ERR_INVALID_ARG                    # no offsets
    assert g(4, BAD + 2, *ok_epi) == bsg.BSG_ERR_MISALIGNED                  # offsets
    assert g(4, BAD, None, None, None, 100, BAD, None) == bsg.BSG_ERR_INVALID_ARG   # m_out != M
    assert g(4, BAD, BAD + 4, None, None, 128, BAD, None) == bsg.BSG_ERR_MISALIGNED  # bias
    assert lib.nvfp4_grouped_gemm(4, 128, 60, 256, BAD, BAD, BAD, BAD, BAD, 1.0, *ok_epi) == \
        bsg.BSG_ERR_INVALID_ARG                                               # N % 8
    s = lib.nvfp4_swizzle_scales_grouped
    assert s(0, 128, 256, BAD, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s(4, 0, 256, BAD, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s(4, 128, 24, BAD, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG       # K % 16
    assert s(4, 128, 256, None, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert s(4, 128, 256, BAD, BAD, BAD + 8, None) == bsg.BSG_ERR_MISALIGNED
    # bound: (ceil(M/128) + E) block rows of 128 x pad4(K/16)
    assert bsg.nvfp4_grouped_scale_bytes(1, 128, 256) == 2 * 128 * 16
    assert bsg.nvfp4_grouped_scale_bytes(3, 300, 1040) == (3 + 3) * 128 * 68
    assert bsg.nvfp4_grouped_scale_bytes(0, 128, 256) == 0
    import oracle
    assert bsg.nvfp4_grouped_scale_bytes(5, 1000, 512) == oracle.get().grouped_scale_bytes(5, 1000, 512)


@pytest.mark.parametrize("entry", ["nvfp4_dense_gemm", "nvfp4_dense_f16_gemm"])
def test_dense_bad_args_and_plans(lib, entry):
    """nvfp4_dense_gemm / nvfp4_dense_f16_gemm: K % 64, N % 8, nulls,
    alignment and the epilogue rules are checked before any launch; the
    planner's dense plans."""
    d = lambda M, N, K, *p: getattr(lib, entry)(M, N, K, *p)  # noqa: E731
    ok = (BAD, BAD, BAD, 1.0, None, None, None)
    assert d(128, 64, 96, *ok, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG        # K % 64
    assert d(128, 60, 128, *ok, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG       # N % 8
    assert d(0, 64, 128, *ok, 0, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert d(128, 64, 128, None, BAD, BAD, 1.0, None, None, None, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert d(128, 64, 128, *ok, 100, BAD, None) == bsg.BSG_ERR_INVALID_ARG       # m_out != M
    assert d(128, 64, 128, BAD, BAD, BAD + 2, 1.0, None, None, None, 128, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert bsg.bsg_select_plan(2, 4096, 4096, 4096, 152) == "nvfp4bf16_tc1_128x256_s5_acc1_tmema"
    assert bsg.bsg_select_plan(2, 128, 4096, 4096, 152) == "nvfp4bf16_tc1_128x256_s5_acc1_tmema"
    assert bsg.bsg_select_plan(2, 4096, 128, 4096, 152) == "nvfp4bf16_tc1_128x128_s8_acc2_tmema"


def test_ingress_probe_bad_args(lib):
    """bsg_measure_ingress checks its arguments before touching the GPU."""
    import ctypes
    out = ctypes.c_double(0.0)
    m = lib.bsg_measure_ingress
    m.argtypes = [ctypes.c_size_t, ctypes.c_int, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                  ctypes.POINTER(ctypes.c_double)]
    assert m(32 << 20, 0, 0, ctypes.byref(out), None) == bsg.BSG_ERR_INVALID_ARG    # stages < 1
    assert m(32 << 20, 7, 0, ctypes.byref(out), None) == bsg.BSG_ERR_INVALID_ARG    # stages > 6
    assert m(64 << 10, 2, 0, ctypes.byref(out), None) == bsg.BSG_ERR_INVALID_ARG    # source < 128 KiB
    assert m(1 << 20, 2, 1, ctypes.byref(out), None) == bsg.BSG_ERR_INVALID_ARG     # boxes need >= 2 MiB
    assert m(32 << 20, 2, 0, None, None) == bsg.BSG_ERR_INVALID_ARG                 # no output


@pytest.mark.parametrize("entry", ["nvfp4_dense_grouped_gemm", "nvfp4_dense_f16_grouped_gemm"])
def test_dense_grouped_bad_args(lib, entry):
    """The routed NVFP4 x dense entries check sizes, slice count, pointers
    and alignment before any launch."""
    f = getattr(lib, entry)
    ok = (BAD, BAD, BAD, BAD, 1.0, None, None, None)
    assert f(2, 128, 64, 96, *ok, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG        # K % 64
    assert f(2, 128, 60, 128, *ok, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG       # N % 8
    assert f(0, 128, 64, 128, *ok, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG       # E < 1
    assert f(1025, 128, 64, 128, *ok, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG    # E > 1024
    assert f(2, 128, 64, 128, BAD, BAD, BAD, None, 1.0, None, None, None, 128, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert f(2, 128, 64, 128, BAD, BAD, BAD, BAD + 2, 1.0, None, None, None, 128, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert f(2, 128, 64, 128, BAD + 8, BAD, BAD, BAD, 1.0, None, None, None, 128, BAD, None) == bsg.BSG_ERR_MISALIGNED


@pytest.mark.parametrize("entry", ["nvfp4_dense_kgrouped_gemm", "nvfp4_dense_f16_kgrouped_gemm"])
def test_dense_kgrouped_bad_args(lib, entry):
    """The K-ragged entries check sizes, slice count, pointers and alignment
    before any launch."""
    f = getattr(lib, entry)
    assert f(2, 128, 64, 96, BAD, BAD, BAD, BAD, 1.0, None, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG   # K % 64
    assert f(2, 128, 60, 128, BAD, BAD, BAD, BAD, 1.0, None, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG  # N % 8
    assert f(0, 128, 64, 128, BAD, BAD, BAD, BAD, 1.0, None, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG  # E < 1
    assert f(2, 128, 64, 128, BAD, BAD, BAD, None, 1.0, None, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG  # no koffs
    assert f(2, 128, 64, 128, BAD, BAD, BAD, BAD + 2, 1.0, None, None, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert f(2, 128, 64, 128, BAD, BAD, BAD, BAD, 1.0, BAD + 4, None, BAD, None) == bsg.BSG_ERR_MISALIGNED  # bias


def test_packed_operand_bytes_and_bad_args(lib):
    """Tile-packed layout: size rule, and argument checks before any launch."""
    assert bsg.nvfp4_packed_operand_bytes(1, 256) == 128 * 128
    assert bsg.nvfp4_packed_operand_bytes(300, 768) == 384 * 384
    assert bsg.nvfp4_packed_operand_bytes(16384, 16384) == 16384 * 8192
    for rows, K in ((0, 256), (8, 128), (8, 384), (-1, 256)):
        assert bsg.nvfp4_packed_operand_bytes(rows, K) == 0
        assert lib.nvfp4_pack_operand(rows, K, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.nvfp4_pack_operand(128 * 65536, 256, BAD, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.nvfp4_pack_operand(8, 256, None, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert lib.nvfp4_pack_operand(8, 256, BAD + 8, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert lib.nvfp4_pack_operand(8, 256, BAD, BAD + 4, None) == bsg.BSG_ERR_MISALIGNED
    g = lib.nvfp4_gemm_packed
    for M, N, K in ((0, 8, 256), (8, 8, 300), (8, 12, 256)):
        assert g(M, N, K, BAD, BAD, BAD, BAD, 1.0, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert g(8, 8, 256, None, BAD, BAD, BAD, 1.0, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert g(8, 8, 256, BAD, BAD, BAD + 8, BAD, 1.0, BAD, None) == bsg.BSG_ERR_MISALIGNED
    ge = lib.nvfp4_gemm_packed_ex
    assert ge(8, 8, 256, BAD, BAD, BAD, BAD, 1.0, None, None, None, 9, BAD, None) == bsg.BSG_ERR_INVALID_ARG
    assert ge(8, 8, 256, BAD, BAD, BAD, BAD, 1.0, BAD + 4, None, None, 8, BAD, None) == bsg.BSG_ERR_MISALIGNED
    assert ge(8, 8, 256, BAD, BAD, BAD, BAD, 1.0, None, None, BAD, 0, BAD, None) == bsg.BSG_ERR_INVALID_ARG


def test_packed_plan_is_listed_but_not_forceable(lib):
    """The tile-packed plan exists, is never chosen by the planner, and a
    forced packed plan is refused by the other entries' planner."""
    bsg.bsg_force_plan("nvfp4_tc2_256x256_s5_acc1_packed")
    try:
        with pytest.raises(bsg.BsgError) as e:
            bsg.bsg_select_plan(0, 16384, 16384, 16384, 152)
        assert e.value.code == bsg.BSG_ERR_NO_PLAN
    finally:
        bsg.bsg_force_plan(None)
    assert bsg.bsg_select_plan(0, 16384, 16384, 16384, 152) == "nvfp4_tc2_256x256_s5_acc1"
