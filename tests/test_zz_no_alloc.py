"""nvfp4_gemm_noalloc: the NVFP4 GEMM for callers that cannot allocate device
memory (its swizzled scales go to a fixed device array inside the library
instead of a cudaMalloc'd workspace).

Called through the C ABI on two calls in a row -- the second smaller than the
first, so stale scratch contents would show -- and compared with the existing
nvfp4_gemm entry point bit for bit (both run the same swizzle and the same
GEMM plan on the same bytes, so any difference is a fault), and with the
oracle's D within the parity tolerance. This file is collected last on purpose.
"""
import numpy as np
import pytest
import torch

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg
import oracle
import workloads

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def test_noalloc_matches_nvfp4_gemm_on_two_calls_in_a_row():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    w = workloads.WORKLOADS["nvfp4_4096"]
    for M, N, K in ((512, 768, 2048), (200, 264, 1024)):
        p = workloads.make_nvfp4(w, "cpu", M=M, N=N, K=K)
        t = {k: p[k].to(dev) for k in ("A", "sfA", "B", "sfB")}
        D_new = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        D_old = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
        bsg.nvfp4_gemm_noalloc(M, N, K, t["A"], t["sfA"], t["B"], t["sfB"], p["alpha"], D_new)
        assert bsg.bsg_last_launch_count() == 2       # the swizzle and the GEMM
        bsg.nvfp4_gemm(M, N, K, t["A"], t["sfA"], t["B"], t["sfB"], p["alpha"], D_old)
        torch.cuda.synchronize()
        assert bsg.bsg_get_device_status() == bsg.BSG_OK
        new, old = _bits(D_new), _bits(D_old)
        assert np.array_equal(new, old), f"{M}x{N}x{K}: {int((new != old).sum())} outputs differ from nvfp4_gemm"
        _, T, Dref = oracle.get().nvfp4_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(),
                                             p["sfB"].numpy(), p["alpha"], K)
        ok = oracle.within_tolerance(new, Dref, T)
        assert ok.all(), f"{M}x{N}x{K}: {int((~ok).sum())} outputs outside tolerance of the oracle"


def test_noalloc_rejects_requests_beyond_its_scratch():
    __graft_entry__.build()
    n = 16384   # 2 x 16 MiB of swizzled scales > the 16 MiB array
    fake = 0x1000
    rc = bsg.load().nvfp4_gemm_noalloc(n, n, n, fake, fake, fake, fake, 1.0, fake, None)
    assert rc == bsg.BSG_ERR_EXCEEDS_SCRATCH
    assert "scratch" in bsg.bsg_error_string(rc)
    assert bsg.bsg_last_launch_count() == 0


def test_noalloc_rejects_misaligned_pointers_before_any_launch():
    """A misaligned operand gets nvfp4_gemm's status, and nothing runs: the
    scratch array and D keep their contents."""
    __graft_entry__.build()
    dev = torch.device("cuda:0")
    M, N, K = 256, 256, 512
    w = workloads.WORKLOADS["nvfp4_4096"]
    p = workloads.make_nvfp4(w, "cpu", M=M, N=N, K=K)
    t = {k: p[k].to(dev) for k in ("A", "sfA", "B", "sfB")}
    D = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    lib = bsg.load()
    a_bad = t["A"].data_ptr() + 8
    for fn in (lib.nvfp4_gemm_noalloc, lib.nvfp4_gemm):
        rc = fn(M, N, K, a_bad, t["sfA"].data_ptr(), t["B"].data_ptr(), t["sfB"].data_ptr(), 1.0,
                D.data_ptr(), None)
        assert rc == bsg.BSG_ERR_MISALIGNED
        assert bsg.bsg_last_launch_count() == 0
    torch.cuda.synchronize()
    assert torch.isnan(D.float()).all()
