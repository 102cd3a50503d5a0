"""Device-side failure detection without a GPU fault: a bounded wait that
nothing completes must give up, report CONV2D_ERR_TIMEOUT with its site
through conv2d_device_status, clear the error word on reading, and leave the
context usable for the next layer call."""
import pytest
import torch

from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.workloads import ACT_TANH, BF16, NORM_BATCH, LayerSpec, random_layer_inputs
from parity_util import check_pair, run_pair

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives():
    assert abi.conv2d_device_status() == (abi.OK, 0)
    abi.check(abi.conv2d_selftest_wait_limit(), "conv2d_selftest_wait_limit")
    rc, site = abi.conv2d_device_status()
    assert (rc, site) == (abi.ERR_TIMEOUT, 6)
    assert abi.conv2d_device_status() == (abi.OK, 0)  # cleared by the read
    spec = LayerSpec(N=2, H=10, W=10, IC=64, OC=64, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_TANH,
                     dtype=BF16)
    gpu, ref = run_pair(spec, random_layer_inputs(spec, 13))
    check_pair(spec, gpu, ref)
