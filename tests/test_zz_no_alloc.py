"""conv2d_fwd_train_noalloc: the training forward for callers that cannot
allocate device memory (their device memory is fixed at start-up, or they
only hold the tensors they pass in). It must give the same results as
conv2d_fwd_train with a caller workspace, call after call, although every
call reuses the library's one static scratch array.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.workloads import (ACT_RELU, ACT_TANH, BF16, FP32, NORM_BATCH, LayerSpec,
                                          random_layer_inputs)
from parity_util import TOL, rel_err, f64

pytestmark = pytest.mark.gpu

CASES = [
    LayerSpec(N=4, H=20, W=20, IC=64, OC=96, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_RELU, dtype=BF16),
    LayerSpec(N=2, H=13, W=11, IC=5, OC=40, KH=3, KW=3, stride=2, pad=1, norm=NORM_BATCH, act=ACT_TANH, dtype=FP32),
]


def _desc(s):
    return abi.desc(s.N, s.H, s.W, s.IC, s.OC, s.KH, s.KW, s.stride, s.pad, s.norm, s.act, s.dtype, s.eps, s.momentum)


def _outputs(spec, dt):
    y_shape = (spec.N, spec.OH, spec.OW, spec.OC)
    f32 = dict(device="cuda", dtype=torch.float32)
    return dict(pre=torch.full(y_shape, 7.0, device="cuda", dtype=dt), y=torch.full(y_shape, 7.0, device="cuda", dtype=dt),
                mean=torch.zeros(spec.OC, **f32), istd=torch.zeros(spec.OC, **f32),
                rm=torch.zeros(spec.OC, **f32), rv=torch.ones(spec.OC, **f32))


@pytest.mark.parametrize("spec", CASES, ids=["bf16_bn_relu", "fp32_bn_tanh_ic5"])
def test_noalloc_matches_workspace_call_twice(spec):
    dt = torch.bfloat16 if spec.dtype == BF16 else torch.float32
    inp = random_layer_inputs(spec, 41)
    li = inp["layers"][0]
    x, w = inp["x"].cuda(), li.w.cuda()
    b, g, bt = li.b.cuda(), li.gamma.cuda(), li.beta.cuda()
    d = _desc(spec)
    ref = _outputs(spec, dt)
    ws = torch.empty(max(abi.conv2d_workspace_size(d, abi.OP_FWD_TRAIN), 256), dtype=torch.uint8, device="cuda")
    abi.check(abi.conv2d_fwd_train(d, x, w, b, g, bt, ref["rm"], ref["rv"], ref["pre"], ref["mean"], ref["istd"],
                                   ref["y"], ws), "conv2d_fwd_train")
    for call in range(2):
        out = _outputs(spec, dt)
        abi.check(abi.conv2d_fwd_train_noalloc(d, x, w, b, g, bt, out["rm"], out["rv"], out["pre"], out["mean"],
                                               out["istd"], out["y"]), "conv2d_fwd_train_noalloc")
        torch.cuda.synchronize()
        assert abi.conv2d_device_status()[0] == abi.OK
        for k in ("pre", "y", "mean", "istd", "rm", "rv"):
            err = rel_err(f64(out[k]), f64(ref[k]))
            assert err <= TOL[spec.dtype], (call, k, err)


def test_noalloc_refuses_specs_beyond_its_scratch():
    # per-tile statistics of a 4096x64x64x256 batch-norm layer need far more than 32 MiB
    big = LayerSpec(N=4096, H=64, W=64, IC=8, OC=256, KH=1, KW=1, norm=NORM_BATCH, act=ACT_RELU, dtype=BF16)
    d = _desc(big)
    assert abi.conv2d_workspace_size(d, abi.OP_FWD_TRAIN) > 32 << 20
    t = torch.zeros(16, device="cuda")
    rc = abi.conv2d_fwd_train_noalloc(d, t, t, None, t, t, t, t, t, t, t, t)
    assert rc == abi.ERR_WORKSPACE
