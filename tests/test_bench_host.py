"""Host-side checks of bench.py's bookkeeping (no GPU)."""
import bench


def test_traffic_constant_matches_kernel_sources():
    """Every DRAM-traffic figure is stored with the digest of the pair
    kernel's sources it was captured on; a kernel change must come with a
    fresh capture (otherwise roofline.traffic reads null)."""
    current = bench.kernel_digest()
    for key, (digest, bytes_) in bench.NCU_TRAFFIC_BYTES.items():
        assert digest == current, f"{key}: traffic captured on kernel {digest}, sources are now {current}"
        assert bytes_ > 0
        assert bench.ncu_traffic(*key) == bytes_


def test_traffic_exceeds_algorithmic_bytes():
    """DRAM traffic of a launch cannot be below its algorithmic bytes: A, B,
    both scale sets and D of the 16384^3 workload."""
    n = 16384
    algorithmic = 2 * n * n // 2 + 2 * n * n // 16 + 2 * n * n
    for (plan, workload), (_, bytes_) in bench.NCU_TRAFFIC_BYTES.items():
        if workload == "nvfp4_16384":
            assert bytes_ >= algorithmic
