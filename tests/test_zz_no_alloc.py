"""conv2d_fwd_train_noalloc: the training forward for callers that cannot
allocate device memory (their device memory is fixed at start-up, or they
only hold the tensors they pass in). It runs the same kernels as
conv2d_fwd_train with a caller workspace, so its results must be bitwise
equal to that call's, call after call, although every call reuses the
library's one static scratch array: a call that left more of the array
written (a larger layer) must not leak into the next, smaller one.

This file is collected last on purpose, so a run that stops at the first
failure has already run every other test."""
import pytest
import torch

from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.workloads import (ACT_RELU, ACT_SIGMOID, ACT_TANH, BF16, FP32, NORM_BATCH, LayerSpec,
                                          random_layer_inputs)

pytestmark = pytest.mark.gpu

CASES = [
    LayerSpec(N=4, H=20, W=20, IC=64, OC=96, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_RELU, dtype=BF16),
    LayerSpec(N=2, H=13, W=11, IC=5, OC=40, KH=3, KW=3, stride=2, pad=1, norm=NORM_BATCH, act=ACT_TANH, dtype=FP32),
]
KEYS = ("pre", "y", "mean", "istd", "rm", "rv")


def _desc(s):
    return abi.desc(s.N, s.H, s.W, s.IC, s.OC, s.KH, s.KW, s.stride, s.pad, s.norm, s.act, s.dtype, s.eps, s.momentum)


def _dt(spec):
    return torch.bfloat16 if spec.dtype == BF16 else torch.float32


def _outputs(spec):
    y_shape = (spec.N, spec.OH, spec.OW, spec.OC)
    f32 = dict(device="cuda", dtype=torch.float32)
    dt = _dt(spec)
    return dict(pre=torch.full(y_shape, 7.0, device="cuda", dtype=dt), y=torch.full(y_shape, 7.0, device="cuda", dtype=dt),
                mean=torch.zeros(spec.OC, **f32), istd=torch.zeros(spec.OC, **f32),
                rm=torch.zeros(spec.OC, **f32), rv=torch.ones(spec.OC, **f32))


def _inputs(spec, seed):
    inp = random_layer_inputs(spec, seed)
    li = inp["layers"][0]
    return (inp["x"].cuda(), li.w.cuda(), li.b.cuda(), li.gamma.cuda(), li.beta.cuda())


def _with_workspace(spec, args):
    """Reference: conv2d_fwd_train with a caller workspace that starts out as garbage (0xFF bytes)."""
    d = _desc(spec)
    out = _outputs(spec)
    ws = torch.full((max(abi.conv2d_workspace_size(d, abi.OP_FWD_TRAIN), 256),), 255, dtype=torch.uint8,
                    device="cuda")
    x, w, b, g, bt = args
    abi.check(abi.conv2d_fwd_train(d, x, w, b, g, bt, out["rm"], out["rv"], out["pre"], out["mean"], out["istd"],
                                   out["y"], ws), "conv2d_fwd_train")
    torch.cuda.synchronize()
    return out


def _noalloc(spec, args):
    d = _desc(spec)
    out = _outputs(spec)
    x, w, b, g, bt = args
    abi.check(abi.conv2d_fwd_train_noalloc(d, x, w, b, g, bt, out["rm"], out["rv"], out["pre"], out["mean"],
                                           out["istd"], out["y"]), "conv2d_fwd_train_noalloc")
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    return out


def _assert_equal(out, ref, where):
    for k in KEYS:
        assert torch.equal(out[k], ref[k]), (where, k, float((out[k].float() - ref[k].float()).abs().max()))


@pytest.mark.parametrize("spec", CASES, ids=["bf16_bn_relu", "fp32_bn_tanh_ic5"])
def test_noalloc_matches_workspace_call_twice(spec):
    args = _inputs(spec, 41)
    ref = _with_workspace(spec, args)
    for call in range(2):
        _assert_equal(_noalloc(spec, args), ref, "call %d" % call)


def test_noalloc_larger_then_smaller_layer():
    """A larger layer fills more of the shared scratch array (packed input, more per-tile statistics); the
    smaller layer that follows must read none of what it left behind."""
    big = LayerSpec(N=6, H=40, W=40, IC=5, OC=96, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_SIGMOID,
                    dtype=FP32)
    small = LayerSpec(N=2, H=9, W=9, IC=5, OC=40, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_SIGMOID,
                      dtype=FP32)
    assert (abi.conv2d_workspace_size(_desc(big), abi.OP_FWD_TRAIN) >
            2 * abi.conv2d_workspace_size(_desc(small), abi.OP_FWD_TRAIN))
    big_args, small_args = _inputs(big, 43), _inputs(small, 44)
    ref_big = _with_workspace(big, big_args)
    ref_small = _with_workspace(small, small_args)
    _assert_equal(_noalloc(big, big_args), ref_big, "large layer")
    _assert_equal(_noalloc(small, small_args), ref_small, "smaller layer after the large one")
    _assert_equal(_noalloc(big, big_args), ref_big, "large layer again")


def test_noalloc_refuses_specs_beyond_its_scratch():
    # per-tile statistics of a 4096x64x64x256 batch-norm layer need far more than 32 MiB
    big = LayerSpec(N=4096, H=64, W=64, IC=8, OC=256, KH=1, KW=1, norm=NORM_BATCH, act=ACT_RELU, dtype=BF16)
    d = _desc(big)
    assert abi.conv2d_workspace_size(d, abi.OP_FWD_TRAIN) > 32 << 20
    t = torch.zeros(16, device="cuda")
    rc = abi.conv2d_fwd_train_noalloc(d, t, t, None, t, t, t, t, t, t, t, t)
    assert rc == abi.ERR_WORKSPACE
