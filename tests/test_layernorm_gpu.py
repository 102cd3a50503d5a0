"""Layer norm on the GPU against the oracle: the pages' third `Normalization`
value, with per-image statistics over OH*OW*OC of the stored pre-activations
(`forward` / `evaluate` LAYER_NORM branches) and the training backward whose
projection sums run over each image (`backward_full`, NORM_DIM = batch).

Cases: the BN-layer and large workload shapes with layer norm at reduced
batch, images spanning several blocks of the walk, two column tiles (the
epilogue's per-tile row partials), channel counts off the vector width (the
unvectorised walk), 1x1 outputs (statistics over OC values only), inference,
accumulation and partial backward, and the full-size large shape checked
through properties.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.layer import Conv2dLayer
from conv2d_layer_gb300.workloads import (ACT_IDENTITY, ACT_RELU, ACT_SIGMOID, ACT_TANH, BF16, FP32, NORM_LAYER,
                                          WORKLOADS, LayerSpec, make_inputs, random_layer_inputs)
from parity_util import TOL, check_pair, f64, oracle_layer, rel_err, run_pair

pytestmark = pytest.mark.gpu


def _wl(name, **over):
    spec = replace(WORKLOADS[name].layers[0], norm=NORM_LAYER, **over)
    return spec, make_inputs(name, layers=[spec])


LN_CASES = {
    "bn_shape_n4_fp32": lambda: _wl("bn", N=4),
    "large_shape_n2_bf16": lambda: _wl("large", N=2, H=28, W=28),
    "bf16_56x56_images_span_blocks": lambda: (lambda s: (s, random_layer_inputs(s, 3)))(
        LayerSpec(N=2, H=56, W=56, IC=64, OC=64, KH=3, KW=3, stride=1, pad=1, norm=NORM_LAYER, act=ACT_TANH,
                  dtype=BF16)),
    "bf16_oc300_two_tiles_sigmoid": lambda: (lambda s: (s, random_layer_inputs(s, 4)))(
        LayerSpec(N=2, H=9, W=9, IC=64, OC=300, KH=3, KW=3, stride=1, pad=1, norm=NORM_LAYER, act=ACT_SIGMOID,
                  dtype=BF16)),
    "fp32_oc136_two_tiles_relu": lambda: (lambda s: (s, random_layer_inputs(s, 5)))(
        LayerSpec(N=2, H=7, W=7, IC=8, OC=136, KH=3, KW=3, stride=1, pad=1, norm=NORM_LAYER, act=ACT_RELU,
                  dtype=FP32)),
    "fp32_oc5_unvectorised_s2": lambda: (lambda s: (s, random_layer_inputs(s, 6)))(
        LayerSpec(N=3, H=10, W=10, IC=3, OC=5, KH=3, KW=3, stride=2, pad=1, norm=NORM_LAYER, act=ACT_RELU,
                  dtype=FP32)),
    "bf16_ic40_oc72_ragged_tanh": lambda: (lambda s: (s, random_layer_inputs(s, 8)))(
        LayerSpec(N=3, H=13, W=13, IC=40, OC=72, KH=3, KW=3, stride=1, pad=1, norm=NORM_LAYER, act=ACT_TANH,
                  dtype=BF16)),
    "bf16_out1x1_identity": lambda: (lambda s: (s, random_layer_inputs(s, 9)))(
        LayerSpec(N=5, H=3, W=3, IC=64, OC=64, KH=3, KW=3, stride=1, pad=0, norm=NORM_LAYER, act=ACT_IDENTITY,
                  dtype=BF16)),
}


@pytest.mark.parametrize("name", list(LN_CASES))
def test_layernorm_parity(name):
    spec, inp = LN_CASES[name]()
    gpu, ref = run_pair(spec, inp)
    assert gpu["mean"].shape == (spec.N,)
    check_pair(spec, gpu, ref)
    # no running statistics under layer norm: the layer's buffers are untouched
    li = inp["layers"][0]
    assert np.array_equal(gpu["running_mean"], f64(li.running_mean))
    assert np.array_equal(gpu["running_var"], f64(li.running_var))


@pytest.mark.parametrize("dtype", [FP32, BF16])
def test_layernorm_accumulate_and_partial_backward(dtype):
    spec = LayerSpec(N=2, H=12, W=12, IC=16, OC=32, KH=3, KW=3, stride=1, pad=1, norm=NORM_LAYER, act=ACT_TANH,
                     dtype=dtype)
    inp = random_layer_inputs(spec, 11)
    gpu, ref = run_pair(spec, inp, prev_grads=True)
    check_pair(spec, gpu, ref)
    gpu, ref = run_pair(spec, inp, need_params=False)
    check_pair(spec, gpu, ref, need_params=False)
    gpu, ref = run_pair(spec, inp, need_dx=False)
    check_pair(spec, gpu, ref, need_dx=False)


@pytest.mark.parametrize("act,dtype", [(ACT_RELU, FP32), (ACT_TANH, BF16)])
def test_layernorm_infer_parity(act, dtype):
    spec = LayerSpec(N=3, H=15, W=15, IC=32, OC=48, KH=3, KW=3, stride=2, pad=1, norm=NORM_LAYER, act=act,
                     dtype=dtype)
    inp = random_layer_inputs(spec, 5)
    li = inp["layers"][0]
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta)
    y = L.fwd_infer(inp["x"].cuda())
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    ref = oracle.fwd_infer(oracle_layer(spec), f64(inp["x"]), f64(li.w), f64(li.b), f64(li.gamma), f64(li.beta))
    assert rel_err(f64(y), ref) <= TOL[dtype]


def test_layernorm_fullsize_large_properties():
    """The large workload shape with layer norm at full size (N=256, 56x56x256, bf16): per-image statistics
    of the stored pre-activations, the normalise + activation relation for every element, dgamma / dbeta as
    their defining sums, and d_conv's per-image sums through dbias (sum over channels of dbias is 0)."""
    spec = replace(WORKLOADS["large"].layers[0], norm=NORM_LAYER)
    inp = make_inputs("large", layers=[spec])
    li = inp["layers"][0]
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    L.zero_grad()
    L.fwd_train(x)
    L.bwd(x, dy)
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    N, C = spec.N, spec.OC
    pre = L.pre_act.double().reshape(N, -1)
    mean_s, var_s = pre.mean(1), pre.var(1, unbiased=False)
    mean_g, istd_g = L.save_mean.double(), L.save_inv_std.double()
    std_s = var_s.sqrt()
    assert torch.all((mean_g - mean_s).abs() <= 1e-5 * std_s), "per-image mean"
    assert torch.all((1.0 / istd_g ** 2 - spec.eps - var_s).abs() <= 1e-5 * var_s), "per-image var"
    g, bt = L.gamma.double(), L.beta.double()
    z = ((pre - mean_g[:, None]) * istd_g[:, None]).reshape(N, -1, C)
    u = g * z + bt
    y_ref = torch.relu(u)
    y_err = (L.y.double().reshape(N, -1, C) - y_ref).abs()
    u8 = 2.0 ** -8
    assert torch.all(y_err <= u8 * y_ref.abs() + 1e-5 * y_ref.abs().max()), "y"
    del y_ref, y_err
    d = dy.double().reshape(N, -1, C)
    dn = (u > 0).double() * d
    near = u.abs() <= 1e-5 * ((g * z).abs() + bt.abs() + 1e-30)
    slack_b = (near * d.abs()).sum((0, 1))
    slack_g = (near * (d * z).abs()).sum((0, 1))
    dbeta_ref, dgamma_ref = dn.sum((0, 1)), (dn * z).sum((0, 1))
    tol = TOL[BF16]
    assert torch.all((L.dbeta.double() - dbeta_ref).abs() <= tol * dbeta_ref.abs().max() + slack_b), "dbeta"
    assert torch.all((L.dgamma.double() - dgamma_ref).abs() <= tol * dgamma_ref.abs().max() + slack_g), "dgamma"
    # d_conv sums to zero over each image, so the channel sum of dbias vanishes against its scale
    db = L.db.double()
    assert abs(float(db.sum())) <= 2e-2 * float(db.abs().sum()) + 1e-6, "sum of dbias"
