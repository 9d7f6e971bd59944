"""The operand-ingress probe on the GPU: it runs clean and reports a rate an
SM can physically sustain (a few to a few hundred bytes per cycle), and the
L2-resident source is at least as fast as one eight times the size of L2."""
from __future__ import annotations

import pytest
import torch

import __graft_entry__
import block_scaled_precision_persistent_gb300 as bsg

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    __graft_entry__.build()
    torch.cuda.set_device(0)
    return torch.device("cuda:0")


def test_ingress_probe(dev):
    l2 = torch.cuda.get_device_properties(0).L2_cache_size
    per_sm_l2, total_l2 = bsg.bsg_measure_ingress(32 << 20, 4)
    per_sm_dram, total_dram = bsg.bsg_measure_ingress(8 * l2, 4)
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert 4.0 < per_sm_l2 < 512.0 and 4.0 < per_sm_dram < 512.0
    assert total_l2 > 1000.0 and total_dram > 1000.0
    assert per_sm_l2 >= 0.9 * per_sm_dram
    per_sm_box, total_box = bsg.bsg_measure_ingress(32 << 20, 4, tensor_boxes=True)
    assert bsg.bsg_get_device_status() == bsg.BSG_OK
    assert 4.0 < per_sm_box < 512.0 and total_box > 1000.0
