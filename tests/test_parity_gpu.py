"""GPU parity: the C-ABI CUDA path against the CPU oracle, element by element,
on the same seeded inputs, at sizes the oracle finishes in seconds that still
span several tiles and a ragged tail; plus the edge cases of the layer
(channel counts that are not a multiple of the vector width, more than one
column tile, 1x1 outputs, strides larger than the kernel, stride-4 dgrad).
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.layer import Conv2dLayer
from conv2d_layer_gb300.workloads import (ACT_IDENTITY, ACT_RELU, ACT_SIGMOID, ACT_TANH, BF16, FP32, NORM_BATCH,
                                          NORM_GROUP, NORM_LAYER, NORM_NONE, WORKLOADS, LayerSpec, make_inputs,
                                          random_layer_inputs)
from parity_util import check_pair, f64, oracle_layer, rel_err, run_pair, TOL

import oracle

pytestmark = pytest.mark.gpu


def _wl(name, **over):
    spec = replace(WORKLOADS[name].layers[0], **over)
    return spec, make_inputs(name, layers=[spec])


CONFIG_CASES = {
    # the five workloads at reduced batch / spatial size (same channels, kernels, strides, modes)
    "tiny": lambda: (WORKLOADS["tiny"].layers[0], make_inputs("tiny")),
    "rl_n3": lambda: _wl("rl", N=3),
    "bn_n4": lambda: _wl("bn", N=4),
    "mixed_l1_20x20": lambda: (lambda s: (s, random_layer_inputs(s, 31)))(
        replace(WORKLOADS["mixed"].layers[0], N=2, H=20, W=20)),
    "mixed_l2_20x20": lambda: (lambda s: (s, random_layer_inputs(s, 32)))(
        replace(WORKLOADS["mixed"].layers[1], N=2, H=20, W=20)),
    "large_20x20": lambda: _wl("large", N=1, H=20, W=20),
}

EDGE_CASES = {
    "bf16_ic3_oc20_k5s3p2_sigmoid": LayerSpec(N=2, H=13, W=13, IC=3, OC=20, KH=5, KW=5, stride=3, pad=2,
                                              norm=NORM_NONE, act=ACT_SIGMOID, dtype=BF16),
    "fp32_ic5_oc130_k3s2p1_bn_tanh": LayerSpec(N=2, H=9, W=9, IC=5, OC=130, KH=3, KW=3, stride=2, pad=1,
                                               norm=NORM_BATCH, act=ACT_TANH, dtype=FP32),
    "bf16_oc320_1x1_identity": LayerSpec(N=3, H=7, W=7, IC=64, OC=320, KH=1, KW=1, stride=1, pad=0,
                                         norm=NORM_NONE, act=ACT_IDENTITY, dtype=BF16),
    "fp32_out1x1_bn_relu": LayerSpec(N=5, H=3, W=3, IC=4, OC=8, KH=3, KW=3, stride=1, pad=0, norm=NORM_BATCH,
                                     act=ACT_RELU, dtype=FP32),
    "bf16_k8s4p2": LayerSpec(N=2, H=36, W=36, IC=8, OC=64, KH=8, KW=8, stride=4, pad=2, norm=NORM_NONE,
                             act=ACT_TANH, dtype=BF16),
    "fp32_k4s2p1_identity": LayerSpec(N=2, H=10, W=10, IC=4, OC=16, KH=4, KW=4, stride=2, pad=1, norm=NORM_NONE,
                                      act=ACT_IDENTITY, dtype=FP32),
    "bf16_ic16_bn_sigmoid": LayerSpec(N=2, H=16, W=16, IC=16, OC=64, KH=3, KW=3, stride=1, pad=1,
                                      norm=NORM_BATCH, act=ACT_SIGMOID, dtype=BF16),
    "fp32_stride_gt_kernel": LayerSpec(N=2, H=9, W=9, IC=4, OC=4, KH=2, KW=2, stride=3, pad=0, norm=NORM_NONE,
                                       act=ACT_IDENTITY, dtype=FP32),
    "fp32_rect_kernel": LayerSpec(N=2, H=11, W=7, IC=8, OC=12, KH=3, KW=1, stride=1, pad=1, norm=NORM_BATCH,
                                  act=ACT_SIGMOID, dtype=FP32),
    # bf16 with 64-channel multiples takes the TMA im2col paths; a rectangular kernel on a non-square
    # image makes the H and W bounding-box corners differ
    "bf16_rect_k3x1_tma": LayerSpec(N=3, H=11, W=7, IC=64, OC=64, KH=3, KW=1, stride=1, pad=1, norm=NORM_BATCH,
                                    act=ACT_TANH, dtype=BF16),
    "bf16_k1x5_s2_tma": LayerSpec(N=2, H=9, W=16, IC=128, OC=96, KH=1, KW=5, stride=2, pad=2, norm=NORM_NONE,
                                  act=ACT_RELU, dtype=BF16),
    # batch statistics over two column tiles (every tile takes its own mean first) with a last
    # row tile of 19 pixels (three of four TMEM lane quarters empty, one partly filled)
    "bf16_oc320_1x1_bn_ragged": LayerSpec(N=3, H=7, W=7, IC=64, OC=320, KH=1, KW=1, stride=1, pad=0,
                                          norm=NORM_BATCH, act=ACT_RELU, dtype=BF16),
    "fp32_oc288_k3_bn_ragged": LayerSpec(N=2, H=10, W=9, IC=8, OC=288, KH=3, KW=3, stride=1, pad=1,
                                         norm=NORM_BATCH, act=ACT_IDENTITY, dtype=FP32),
    # stride-2 dgrad with d_conv by TMA, one im2col map per stride phase (ragged phase grids; 2 x 2 taps
    # in every phase of the 4 x 4 kernel)
    "bf16_s2_tma_phases": LayerSpec(N=2, H=13, W=11, IC=64, OC=128, KH=3, KW=3, stride=2, pad=1,
                                    norm=NORM_BATCH, act=ACT_RELU, dtype=BF16),
    "bf16_k4s2_tma_phases": LayerSpec(N=2, H=10, W=10, IC=64, OC=64, KH=4, KW=4, stride=2, pad=1,
                                      norm=NORM_NONE, act=ACT_TANH, dtype=BF16),
    # stride-2 dgrad reading the weights directly as an MN-major operand: three 64-channel groups per tile
    "bf16_s2_weights_mn_ic192": LayerSpec(N=2, H=12, W=10, IC=192, OC=128, KH=3, KW=3, stride=2, pad=1,
                                          norm=NORM_BATCH, act=ACT_RELU, dtype=BF16),
    # the same with four stride phases of 1156 rows each (ten m-tiles, the last with 4 rows)
    "bf16_s2_pair_phases": LayerSpec(N=4, H=34, W=34, IC=64, OC=64, KH=3, KW=3, stride=2, pad=1,
                                     norm=NORM_BATCH, act=ACT_RELU, dtype=BF16),
    # batch-norm backward with d_conv formed inside the dgrad and wgrad producers (1x1, stride 1, bf16,
    # sigmoid): a ragged pixel count (three 128-row tiles and 45 rows; six 64-pixel k-blocks and 45) and a
    # weight-gradient column tile half outside the 192 channels
    "bf16_fused_bwd_sigmoid_ragged": LayerSpec(N=3, H=13, W=11, IC=64, OC=192, KH=1, KW=1, stride=1, pad=0,
                                               norm=NORM_BATCH, act=ACT_SIGMOID, dtype=BF16),
    # fp32 with KW * IC = 32 and no padding: X through the folded im2col view (each kernel row one
    # 32-float run) in the fprop and the weight gradient, at strides 2 and 1
    "fp32_fold_k8_s2": LayerSpec(N=2, H=20, W=21, IC=4, OC=16, KH=8, KW=8, stride=2, pad=0,
                                 norm=NORM_NONE, act=ACT_RELU, dtype=FP32),
    "fp32_fold_k4x8_s1_bn": LayerSpec(N=2, H=9, W=13, IC=4, OC=40, KH=4, KW=8, stride=1, pad=0,
                                      norm=NORM_BATCH, act=ACT_SIGMOID, dtype=FP32),
    # deep fp32 K loops: the accumulation is split over TMEM chunks (dgrad K = 5184, fprop K = 2304)
    "fp32_deep_dgrad_oc576": LayerSpec(N=2, H=10, W=9, IC=8, OC=576, KH=3, KW=3, stride=1, pad=1,
                                       norm=NORM_BATCH, act=ACT_IDENTITY, dtype=FP32),
    "fp32_deep_fprop_ic256": LayerSpec(N=2, H=9, W=9, IC=256, OC=40, KH=3, KW=3, stride=1, pad=1,
                                       norm=NORM_NONE, act=ACT_RELU, dtype=FP32),
    # fp32 with A in tensor memory: three 64-column tiles of the fprop and of the weight gradient with
    # batch statistics per row tile; a stride-2 dgrad with four stride phases; a K loop of 1152 over two
    # accumulator chunks (32-column tiles)
    "fp32_ts_ic32_oc160_bn": LayerSpec(N=2, H=12, W=10, IC=32, OC=160, KH=3, KW=3, stride=1, pad=1,
                                       norm=NORM_BATCH, act=ACT_SIGMOID, dtype=FP32),
    "fp32_ts_s2_phases": LayerSpec(N=2, H=13, W=11, IC=32, OC=64, KH=3, KW=3, stride=2, pad=1, norm=NORM_BATCH,
                                   act=ACT_RELU, dtype=FP32),
    "fp32_ts_two_chunks": LayerSpec(N=2, H=9, W=9, IC=128, OC=40, KH=3, KW=3, stride=1, pad=1, norm=NORM_NONE,
                                    act=ACT_RELU, dtype=FP32),
    # phase-merged dgrad (kernel and padding multiples of the stride: every stride phase in the columns of
    # one GEMM over the coarse grid, stored as runs of S * IC values): bf16 with padding 2 at stride 2, and
    # fp32 at stride 4 with padding 4 and an input whose last coarse row and column are partly outside
    "bf16_merged_k4s2p2": LayerSpec(N=2, H=11, W=13, IC=8, OC=64, KH=4, KW=4, stride=2, pad=2, norm=NORM_BATCH,
                                    act=ACT_TANH, dtype=BF16),
    "fp32_merged_k8s4p4_ragged": LayerSpec(N=2, H=18, W=17, IC=4, OC=32, KH=8, KW=8, stride=4, pad=4,
                                           norm=NORM_NONE, act=ACT_RELU, dtype=FP32),
    # 48 weight-gradient splits (fp32 caps a split at 32 k-blocks; 49152 pixels) with a channel count off
    # the vector width: the split-group reduce with one channel per thread
    "fp32_ic3_many_wgrad_splits": LayerSpec(N=12, H=64, W=64, IC=3, OC=8, KH=3, KW=3, stride=1, pad=1,
                                            norm=NORM_NONE, act=ACT_RELU, dtype=FP32),
}


@pytest.mark.parametrize("name", list(CONFIG_CASES))
def test_config_parity(name):
    spec, inp = CONFIG_CASES[name]()
    gpu, ref = run_pair(spec, inp)
    check_pair(spec, gpu, ref)


@pytest.mark.parametrize("name", list(EDGE_CASES))
def test_edge_parity(name):
    spec = EDGE_CASES[name]
    inp = random_layer_inputs(spec, 7)
    gpu, ref = run_pair(spec, inp)
    check_pair(spec, gpu, ref)


@pytest.mark.parametrize("dtype,norm", [(BF16, NORM_BATCH), (BF16, NORM_LAYER), (BF16, NORM_GROUP),
                                        (FP32, NORM_BATCH)])
def test_signed_gamma_relu(dtype, norm):
    """ReLU after a norm whose gain is positive, negative or zero by channel. The backward's ReLU test
    (on bf16, a packed compare of the stored pre-activation with a key per channel) must follow the
    sign of gamma, and a zero gain leaves the decision to beta alone (both signs of beta present)."""
    spec = LayerSpec(N=2, H=12, W=12, IC=64, OC=64, KH=3, KW=3, stride=1, pad=1, norm=norm,
                     groups=8 if norm == NORM_GROUP else 1, act=ACT_RELU, dtype=dtype)
    inp = random_layer_inputs(spec, 11)
    li = inp["layers"][0]
    c = torch.arange(spec.OC)
    gamma, beta = li.gamma.clone(), li.beta.clone()
    gamma[c % 4 == 1] *= -1.0
    gamma[c % 4 == 3] = 0.0
    beta[c % 8 == 3] = 0.3
    beta[c % 8 == 7] = -0.3
    inp["layers"][0] = replace(li, gamma=gamma, beta=beta)
    gpu, ref = run_pair(spec, inp)
    check_pair(spec, gpu, ref)
    # the zero-gain channels put out beta (beta > 0) or nothing (beta < 0) at every pixel
    assert np.all(ref["y"][..., 3::8] == float(np.float32(0.3))) and np.all(ref["y"][..., 7::8] == 0.0)


@pytest.mark.parametrize("dtype,k", [(FP32, 3), (BF16, 3), (BF16, 1)])
def test_accumulate_and_partial_backward(dtype, k):
    """dW/dbias/dgamma/dbeta accumulate into existing values; dx is overwritten;
    backward_input (params NULL) and backward (dx NULL) variants. The bf16 1x1 layer (64 -> 128 channels)
    takes the backward that forms d_conv inside the GEMM producers."""
    spec = LayerSpec(N=2, H=12, W=12, IC=16 if k == 3 else 64, OC=32 if k == 3 else 128, KH=k, KW=k, stride=1,
                     pad=k // 2, norm=NORM_BATCH, act=ACT_TANH, dtype=dtype)
    inp = random_layer_inputs(spec, 11)
    gpu, ref = run_pair(spec, inp, prev_grads=True)
    check_pair(spec, gpu, ref)
    gpu, ref = run_pair(spec, inp, need_params=False)
    check_pair(spec, gpu, ref, need_params=False)
    gpu, ref = run_pair(spec, inp, need_dx=False)
    check_pair(spec, gpu, ref, need_dx=False)


@pytest.mark.parametrize("norm,act,dtype", [(NORM_BATCH, ACT_RELU, FP32), (NORM_NONE, ACT_SIGMOID, FP32),
                                            (NORM_BATCH, ACT_TANH, BF16), (NORM_NONE, ACT_RELU, BF16)])
def test_infer_parity(norm, act, dtype):
    spec = LayerSpec(N=3, H=15, W=15, IC=32, OC=48, KH=3, KW=3, stride=2, pad=1, norm=norm, act=act, dtype=dtype)
    inp = random_layer_inputs(spec, 5)
    li = inp["layers"][0]
    g = torch.Generator().manual_seed(5)
    rm = torch.randn(spec.OC, generator=g) * 0.2
    rv = torch.rand(spec.OC, generator=g) + 0.5
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta, rm, rv)
    y = L.fwd_infer(inp["x"].cuda())
    torch.cuda.synchronize()
    ref = oracle.fwd_infer(oracle_layer(spec), f64(inp["x"]), f64(li.w), f64(li.b), f64(li.gamma), f64(li.beta),
                           f64(rm), f64(rv))
    assert rel_err(f64(y), ref) <= TOL[dtype]
    # no state written by inference
    assert torch.equal(L.running_mean.cpu(), rm.float()) and torch.equal(L.running_var.cpu(), rv.float())


def test_deterministic_bitwise():
    spec = LayerSpec(N=4, H=16, W=16, IC=32, OC=64, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_RELU,
                     dtype=BF16)
    inp = random_layer_inputs(spec, 3)
    li = inp["layers"][0]
    outs = []
    for _ in range(2):
        L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta)
        x, dy = inp["x"].cuda(), inp["dy"].cuda()
        L.zero_grad()
        L.fwd_train(x)
        L.bwd(x, dy)
        torch.cuda.synchronize()
        outs.append([t.clone() for t in (L.y, L.dx, L.dw, L.db, L.dgamma, L.dbeta, L.running_var)])
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_outputs_stay_inside_their_buffers():
    """Canary-filled guard regions before and after every output stay intact."""
    spec = EDGE_CASES["bf16_ic3_oc20_k5s3p2_sigmoid"]
    spec = replace(spec, norm=NORM_BATCH)
    inp = random_layer_inputs(spec, 9)
    li = inp["layers"][0]
    d = abi.desc(spec.N, spec.H, spec.W, spec.IC, spec.OC, spec.KH, spec.KW, spec.stride, spec.pad, spec.norm,
                 spec.act, spec.dtype, spec.eps, spec.momentum)
    G = 256  # guard elements on each side (keeps 16-byte alignment)

    def guarded(n, dtype, fill):
        buf = torch.full((n + 2 * G,), fill, dtype=dtype, device="cuda")
        return buf, buf[G:G + n]

    y_shape = spec.N * spec.OH * spec.OW * spec.OC
    bufs = {}
    bufs["pre"], pre = guarded(y_shape, torch.bfloat16, 7.0)
    bufs["y"], y = guarded(y_shape, torch.bfloat16, 7.0)
    bufs["dx"], dx = guarded(spec.N * spec.H * spec.W * spec.IC, torch.bfloat16, 7.0)
    bufs["dw"], dw = guarded(spec.OC * spec.KH * spec.KW * spec.IC, torch.float32, 0.0)
    small = {}
    for k in ("db", "dg", "dbt", "mean", "istd", "rm", "rv"):
        bufs[k], small[k] = guarded(spec.OC, torch.float32, 0.0)
    small["rv"].fill_(1.0)
    ws_n = max(abi.conv2d_workspace_size(d, op) for op in range(3))
    ws = torch.empty(ws_n, dtype=torch.uint8, device="cuda")
    x, dyv = inp["x"].cuda(), inp["dy"].cuda()
    w, b = li.w.cuda(), li.b.cuda()
    gm, bt = li.gamma.cuda(), li.beta.cuda()
    abi.check(abi.conv2d_fwd_train(d, x, w, b, gm, bt, small["rm"], small["rv"], pre, small["mean"],
                                   small["istd"], y, ws))
    abi.check(abi.conv2d_bwd(d, x, w, gm, bt, pre, small["mean"], small["istd"], dyv, dx, dw, small["db"],
                             small["dg"], small["dbt"], ws))
    torch.cuda.synchronize()
    for k, buf in bufs.items():
        fill = 7.0 if buf.dtype == torch.bfloat16 else 0.0
        head, tail = buf[:G].float().cpu(), buf[-G:].float().cpu()
        assert torch.all(head == fill) and torch.all(tail == fill), k


def test_device_status_clean():
    rc, site = abi.conv2d_device_status()
    assert rc == abi.OK and site == 0


def test_mixed_two_layer_chain():
    """The mixed workload as a stack: layer 1's output (stored in bf16) feeds layer 2; layer 2's dX
    (stored in bf16) is layer 1's dY. Every output of both layers against the oracle run the same way."""
    specs = [replace(WORKLOADS["mixed"].layers[0], N=2, H=20, W=20),
             replace(WORKLOADS["mixed"].layers[1], N=2, H=20, W=20)]
    inp = make_inputs("mixed", layers=specs)
    l1, l2 = inp["layers"]
    L1 = Conv2dLayer(specs[0], l1.w, l1.b, l1.gamma, l1.beta)
    L2 = Conv2dLayer(specs[1], l2.w, l2.b, l2.gamma, l2.beta)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    L1.zero_grad()
    L2.zero_grad()
    y1 = L1.fwd_train(x)
    L2.fwd_train(y1)
    dx2 = L2.bwd(y1, dy)
    L1.bwd(x, dx2)
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK

    O1, O2 = oracle_layer(specs[0]), oracle_layer(specs[1])
    f1 = oracle.fwd_train(O1, f64(inp["x"]), f64(l1.w), f64(l1.b), f64(l1.gamma), f64(l1.beta))
    y1r = oracle.store_round("bf16", f1["y"])
    f2 = oracle.fwd_train(O2, y1r, f64(l2.w), f64(l2.b), f64(l2.gamma), f64(l2.beta))
    g2 = oracle.bwd(O2, y1r, f64(l2.w), f2["ypre"], f64(inp["dy"]), f64(l2.gamma), f64(l2.beta), f2["mean"],
                    f2["inv_std"])
    dx2r = oracle.store_round("bf16", g2["dx"])
    g1 = oracle.bwd(O1, f64(inp["x"]), f64(l1.w), f1["ypre"], dx2r, f64(l1.gamma), f64(l1.beta), f1["mean"],
                    f1["inv_std"])
    tol = TOL[BF16]
    checks = {"y1": (y1, f1["y"]), "y2": (L2.y, f2["y"]), "dx2": (dx2, g2["dx"]), "dw2": (L2.dw, g2["dw"]),
              "dgamma2": (L2.dgamma, g2["dgamma"]), "dbeta2": (L2.dbeta, g2["dbeta"]), "dx1": (L1.dx, g1["dx"]),
              "dw1": (L1.dw, g1["dw"]), "dgamma1": (L1.dgamma, g1["dgamma"]), "dbeta1": (L1.dbeta, g1["dbeta"])}
    errs = {k: rel_err(f64(a), b) for k, (a, b) in checks.items()}
    assert all(v <= tol for v in errs.values()), errs
    # layer 1 sees the shared seeded input: running statistics to 1e-5. Layer 2's input is layer 1's
    # bf16 output, whose values next to a bf16 rounding midpoint may round either way on either side,
    # so its statistics get the BF16 tensor bar.
    for L, f, t in ((L1, f1, 1e-5), (L2, f2, tol)):
        assert rel_err(f64(L.running_mean), f["running_mean"]) <= t
        assert rel_err(f64(L.running_var), f["running_var"]) <= t


EVAL_CASES = {
    "fp32_relu_s1": LayerSpec(N=3, H=12, W=12, IC=16, OC=32, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH,
                              act=ACT_RELU, dtype=FP32, bn_eval=1),
    "bf16_tanh_s2": LayerSpec(N=2, H=17, W=15, IC=64, OC=96, KH=3, KW=3, stride=2, pad=1, norm=NORM_BATCH,
                              act=ACT_TANH, dtype=BF16, bn_eval=1),
    "bf16_sigmoid_1x1": LayerSpec(N=4, H=9, W=9, IC=128, OC=64, KH=1, KW=1, stride=1, pad=0, norm=NORM_BATCH,
                                  act=ACT_SIGMOID, dtype=BF16, bn_eval=1),
}


@pytest.mark.parametrize("name", list(EVAL_CASES))
def test_eval_mode_batchnorm_parity(name):
    """Batch norm in evaluation mode inside training: running statistics used and left unchanged, the
    frozen-statistics backward."""
    spec = EVAL_CASES[name]
    inp = random_layer_inputs(spec, 19)
    li = inp["layers"][0]
    g = torch.Generator().manual_seed(19)
    li.running_mean = torch.randn(spec.OC, generator=g) * 0.3
    li.running_var = torch.rand(spec.OC, generator=g) + 0.5
    gpu, ref = run_pair(spec, inp)
    check_pair(spec, gpu, ref)
    np.testing.assert_array_equal(gpu["running_mean"], f64(li.running_mean))
    np.testing.assert_array_equal(gpu["running_var"], f64(li.running_var))
