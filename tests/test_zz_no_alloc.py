"""nvfp4_gemm_noalloc: the NVFP4 GEMM for callers that cannot allocate device
memory (its swizzled scales go to a fixed device array inside the library
instead of a cudaMalloc'd workspace).

Called through the C ABI and compared with the existing nvfp4_gemm entry
point, under the parity tolerance of the other tests, on two calls in a row:
the second call is smaller than the first, so stale scratch contents would
show. This file is collected last on purpose.
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
        bsg.nvfp4_gemm(M, N, K, t["A"], t["sfA"], t["B"], t["sfB"], p["alpha"], D_old)
        torch.cuda.synchronize()
        assert bsg.bsg_get_device_status() == bsg.BSG_OK
        _, T, _ = oracle.get().nvfp4_gemm(p["A"].numpy(), p["sfA"].numpy(), p["B"].numpy(),
                                          p["sfB"].numpy(), p["alpha"], K)
        new, old = _bits(D_new), _bits(D_old)
        ok = oracle.within_tolerance(new, old, T)
        assert ok.all(), f"{M}x{N}x{K}: {int((~ok).sum())} outputs differ beyond tolerance"


def test_noalloc_rejects_requests_beyond_its_scratch():
    __graft_entry__.build()
    n = 16384   # 2 x 16 MiB of swizzled scales > the 16 MiB array
    fake = 0x1000
    rc = bsg.load().nvfp4_gemm_noalloc(n, n, n, fake, fake, fake, fake, 1.0, fake, None)
    assert rc == bsg.BSG_ERR_EXCEEDS_SCRATCH
    assert "scratch" in bsg.bsg_error_string(rc)
