"""Group norm on the GPU against the oracle: G groups of OC/G consecutive channels, statistics per
(image, group) of the stored pre-activations, backward as the GroupNorm backward of the WebGPU page
("groupnorm_backward.wgsl") with the activation derivative in front and per-channel dgamma / dbeta.

Cases: the large shape with 32 groups (8 channels a group, one per thread vector) and the BN-layer
shape with 4 groups, images spanning several walk blocks, 3 groups of 32 channels, a channel count
off the vector width (the unvectorised walk), one channel per group (instance norm), one group (layer
norm), accumulation and partial backward, inference, and the full-size large shape with 32 groups
checked through its per-(image, group) statistics.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.layer import Conv2dLayer
from conv2d_layer_gb300.workloads import (ACT_IDENTITY, ACT_RELU, ACT_SIGMOID, ACT_TANH, BF16, FP32, NORM_GROUP,
                                          WORKLOADS, LayerSpec, make_inputs, random_layer_inputs)
from parity_util import TOL, check_pair, f64, oracle_layer, rel_err, run_pair

pytestmark = pytest.mark.gpu


def _wl(name, groups, **over):
    spec = replace(WORKLOADS[name].layers[0], norm=NORM_GROUP, groups=groups, **over)
    return spec, make_inputs(name, layers=[spec])


def _spec(seed, **kw):
    spec = LayerSpec(norm=NORM_GROUP, **kw)
    return spec, random_layer_inputs(spec, seed)


GN_CASES = {
    "large_shape_n2_g32_bf16": lambda: _wl("large", 32, N=2, H=28, W=28),
    "bn_shape_n4_g4_fp32": lambda: _wl("bn", 4, N=4),
    "bf16_56x56_g3_images_span_blocks": lambda: _spec(3, N=2, H=56, W=56, IC=64, OC=96, KH=3, KW=3, stride=1,
                                                      pad=1, act=ACT_TANH, dtype=BF16, groups=3),
    "fp32_oc6_g3_unvectorised": lambda: _spec(4, N=3, H=10, W=10, IC=3, OC=6, KH=3, KW=3, stride=2, pad=1,
                                              act=ACT_RELU, dtype=FP32, groups=3),
    "bf16_g64_instance_norm": lambda: _spec(5, N=3, H=12, W=12, IC=64, OC=64, KH=3, KW=3, stride=1, pad=1,
                                            act=ACT_SIGMOID, dtype=BF16, groups=64),
    "fp32_g1_layer_norm": lambda: _spec(6, N=2, H=9, W=9, IC=8, OC=40, KH=3, KW=3, stride=1, pad=1,
                                        act=ACT_IDENTITY, dtype=FP32, groups=1),
    "bf16_oc300_g10_two_tiles": lambda: _spec(7, N=2, H=9, W=9, IC=64, OC=300, KH=3, KW=3, stride=1, pad=1,
                                              act=ACT_RELU, dtype=BF16, groups=10),
}


@pytest.mark.parametrize("name", list(GN_CASES))
def test_groupnorm_parity(name):
    spec, inp = GN_CASES[name]()
    gpu, ref = run_pair(spec, inp)
    assert gpu["mean"].shape == (spec.N * spec.groups,)
    check_pair(spec, gpu, ref)
    li = inp["layers"][0]
    assert np.array_equal(gpu["running_mean"], f64(li.running_mean))
    assert np.array_equal(gpu["running_var"], f64(li.running_var))


@pytest.mark.parametrize("dtype", [FP32, BF16])
def test_groupnorm_accumulate_and_partial_backward(dtype):
    spec = LayerSpec(N=2, H=12, W=12, IC=16, OC=32, KH=3, KW=3, stride=1, pad=1, norm=NORM_GROUP, groups=8,
                     act=ACT_TANH, dtype=dtype)
    inp = random_layer_inputs(spec, 11)
    gpu, ref = run_pair(spec, inp, prev_grads=True)
    check_pair(spec, gpu, ref)
    gpu, ref = run_pair(spec, inp, need_params=False)
    check_pair(spec, gpu, ref, need_params=False)
    gpu, ref = run_pair(spec, inp, need_dx=False)
    check_pair(spec, gpu, ref, need_dx=False)


@pytest.mark.parametrize("act,dtype", [(ACT_RELU, FP32), (ACT_TANH, BF16)])
def test_groupnorm_infer_parity(act, dtype):
    spec = LayerSpec(N=3, H=15, W=15, IC=32, OC=48, KH=3, KW=3, stride=2, pad=1, norm=NORM_GROUP, groups=6,
                     act=act, dtype=dtype)
    inp = random_layer_inputs(spec, 5)
    li = inp["layers"][0]
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta)
    y = L.fwd_infer(inp["x"].cuda())
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    ref = oracle.fwd_infer(oracle_layer(spec), f64(inp["x"]), f64(li.w), f64(li.b), f64(li.gamma), f64(li.beta))
    assert rel_err(f64(y), ref) <= TOL[dtype]


def test_groupnorm_fullsize_large_statistics():
    """The large shape with 32 groups at full size (N=256, 56x56x256, bf16): the saved per-(image, group)
    statistics against those of the stored pre-activations, and the normalise relation for every element."""
    spec = replace(WORKLOADS["large"].layers[0], norm=NORM_GROUP, groups=32)
    inp = make_inputs("large", layers=[spec])
    li = inp["layers"][0]
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    L.zero_grad()
    L.fwd_train(x)
    L.bwd(x, dy)
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    N, C, G = spec.N, spec.OC, spec.groups
    pre = L.pre_act.double().reshape(N, -1, G, C // G)
    grp = pre.permute(0, 2, 1, 3).reshape(N * G, -1)
    mean_s, var_s = grp.mean(1), grp.var(1, unbiased=False)
    mean_g, istd_g = L.save_mean.double(), L.save_inv_std.double()
    assert torch.all((mean_g - mean_s).abs() <= 1e-5 * var_s.sqrt()), "per-group mean"
    assert torch.all((1.0 / istd_g ** 2 - spec.eps - var_s).abs() <= 1e-5 * var_s), "per-group var"
    m = mean_g.reshape(N, 1, G, 1)
    s = istd_g.reshape(N, 1, G, 1)
    u = (L.gamma.double().reshape(G, C // G) * ((pre - m) * s) + L.beta.double().reshape(G, C // G))
    y_ref = torch.relu(u)
    y_err = (L.y.double().reshape(N, -1, G, C // G) - y_ref).abs()
    assert torch.all(y_err <= 2.0 ** -8 * y_ref.abs() + 1e-5 * y_ref.abs().max()), "y"
