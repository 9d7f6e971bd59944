"""Host-side checks of the seeded input generators (no GPU)."""
import numpy as np
import torch

import workloads


def test_e2m1_encode_ties_and_saturation():
    v = torch.tensor([0.0, 0.25, 0.26, 0.75, 1.25, 1.3, 1.75, 2.5, 2.6, 3.5, 5.0, 5.1, 100.0,
                      -0.75, -7.0, -0.1])
    want = [0, 0, 1, 2, 2, 3, 4, 4, 5, 6, 6, 7, 7, 8 | 2, 8 | 7, 8 | 0]
    assert workloads.e2m1_encode(v).tolist() == want


def test_pack_unpack_roundtrip():
    codes = torch.randint(0, 16, (5, 64), dtype=torch.int32).to(torch.uint8)
    p = workloads.pack_e2m1(codes)
    assert p.shape == (5, 32)
    assert int(p[0, 0]) == int(codes[0, 0]) | (int(codes[0, 1]) << 4)
    assert torch.equal(workloads.unpack_e2m1(p), codes)


def test_generators_are_seeded():
    w = workloads.WORKLOADS["nvfp4_4096"]
    a = workloads.make_nvfp4(w, "cpu", M=64, N=32, K=256)
    b = workloads.make_nvfp4(w, "cpu", M=64, N=32, K=256)
    for k in ("A", "sfA", "B", "sfB"):
        assert torch.equal(a[k], b[k])
    assert a["alpha"] == b["alpha"] and a["alpha"] > 0
    w1 = workloads.WORKLOADS["nvfp4_256"]
    c = workloads.make_nvfp4(w1, "cpu")
    assert c["A"].shape == (256, 128) and c["sfA"].shape == (256, 16) and c["alpha"] == 1.0
    # 2^u scales with u in [-4, 4]: exponent fields 3..11, mantissa 0
    sf = c["sfA"].numpy()
    assert set(np.unique(sf >> 3).tolist()) <= set(range(3, 12)) and not (sf & 7).any()


def test_quantised_scales_are_finite_and_unsigned():
    w = workloads.WORKLOADS["nvfp4_skinny_m64_n3072_k3072"]
    p = workloads.make_nvfp4(w, "cpu", M=64, N=128, K=512)
    for k in ("sfA", "sfB"):
        sf = p[k].numpy()
        assert not (sf & 0x80).any()                  # never sign-set
        assert not ((sf & 0x7F) == 0x7F).any()        # never NaN
        assert (sf > 0).mean() > 0.99                 # two-level scheme keeps them normal-ish
    # dequantised values track the source within the NVFP4 grid
    x = workloads.normal_bf16(64, 512, workloads.seed_for(w, 0), w.std, "cpu")
    codes = workloads.unpack_e2m1(p["A"]).to(torch.int64)
    tab = torch.tensor([0, .5, 1, 1.5, 2, 3, 4, 6, -0., -.5, -1, -1.5, -2, -3, -4, -6],
                       dtype=torch.float64)
    sf = p["sfA"].view(torch.float8_e4m3fn).to(torch.float64).repeat_interleave(16, 1)
    sga = 448.0 * 6.0 / float(x.abs().max())
    deq = tab[codes] * sf / sga
    err = (deq - x.double()).abs().max()
    assert float(err) < 0.25 * float(x.abs().max())


def test_fp8_generator():
    w = workloads.WORKLOADS["fp8_8192"]
    p = workloads.make_fp8(w, "cpu", M=32, N=16, K=128)
    assert p["A"].dtype == torch.uint8 and p["A"].shape == (32, 128)
    a = p["A"].numpy()
    assert not ((a & 0x7F) == 0x7F).any()
    assert p["alpha"] > 0


def test_workload_table():
    names = list(workloads.WORKLOADS)
    assert names[:4] == ["nvfp4_256", "nvfp4_4096", "nvfp4_16384", "fp8_8192"]
    assert len(names) == 4 + 12
    w = workloads.WORKLOADS["nvfp4_16384"]
    assert w.flops == 2 * 16384 ** 3
    assert w.algorithmic_bytes == 2 * 16384 * 16384 * 9 / 16 + 2 * 16384 * 16384
