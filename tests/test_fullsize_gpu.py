"""Full-size checks on the GPU for the RL-encoder, BN, mixed (both layers) and
large workloads, with the same ABI calls and launch configuration as bench.py.

The oracle cannot finish these sizes whole, so two kinds of check are made:
  * the tensor-core paths (fprop, dgrad, wgrad, dbias) at full size with
    identity activation and no norm (same shapes, tiles, grids and splits as
    the real layer), against oracle values computed one by one from the
    original inputs at random sample points;
  * the real layer (batch norm + activation) against properties that hold at
    any size: batch statistics of the stored pre-activations (within the
    storage-rounding bound), the running-statistics update, the normalise +
    activation relation for every element, dgamma / dbeta as the sums their
    definitions give (with an allowance for ReLU inputs so close to 0 that
    either side of the kink is a correct result), and dbias ~ 0 under BN.
"""
from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.layer import Conv2dLayer
from conv2d_layer_gb300.workloads import (ACT_IDENTITY, BF16, NORM_BATCH, NORM_NONE, WORKLOADS, make_inputs,
                                          random_layer_inputs)
from parity_util import TOL, oracle_layer

pytestmark = pytest.mark.gpu

CASES = ["rl", "bn", "mixed_l1", "mixed_l2", "large"]


def _case(name):
    if name == "mixed_l1":
        spec = WORKLOADS["mixed"].layers[0]
        return spec, random_layer_inputs(spec, 3)
    if name == "mixed_l2":
        spec = WORKLOADS["mixed"].layers[1]
        return spec, random_layer_inputs(spec, 33)
    return WORKLOADS[name].layers[0], make_inputs(name)


def _f64(t):
    return t.detach().to("cpu", torch.float64).contiguous().numpy()


@pytest.mark.parametrize("name", CASES)
def test_fullsize_gemm_paths_sampled(name):
    spec0, inp = _case(name)
    spec = replace(spec0, norm=NORM_NONE, act=ACT_IDENTITY)
    li = inp["layers"][0]
    L = Conv2dLayer(spec, li.w, li.b)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    L.zero_grad()
    L.fwd_train(x)
    L.bwd(x, dy)
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    tol = TOL[spec.dtype]
    OL = oracle_layer(spec)
    x64, w64, b64, dy64 = _f64(inp["x"]), _f64(li.w), _f64(li.b), _f64(inp["dy"])
    rng = np.random.default_rng(17)
    ns = 96

    # Ypre at random output elements
    pts = np.stack([rng.integers(0, s, ns) for s in (spec.N, spec.OH, spec.OW, spec.OC)], 1)
    got = L.pre_act[tuple(torch.from_numpy(pts[:, i]).cuda() for i in range(4))].double().cpu().numpy()
    ref = np.array([oracle.conv_point(OL, x64, w64, b64, *map(int, p)) for p in pts])
    assert np.max(np.abs(got - ref)) <= tol * np.max(np.abs(ref)), "ypre"

    # dX at random input elements (identity activation, no norm: d_conv = dY)
    pts = np.stack([rng.integers(0, s, ns) for s in (spec.N, spec.H, spec.W, spec.IC)], 1)
    got = L.dx[tuple(torch.from_numpy(pts[:, i]).cuda() for i in range(4))].double().cpu().numpy()
    ref = np.array([oracle.dgrad_point(OL, dy64, w64, *map(int, p)) for p in pts])
    assert np.max(np.abs(got - ref)) <= tol * np.max(np.abs(ref)), "dx"

    # dW at random weight elements (sums over the whole batch)
    pts = np.stack([rng.integers(0, s, 24) for s in (spec.OC, spec.KH, spec.KW, spec.IC)], 1)
    got = L.dw[tuple(torch.from_numpy(pts[:, i]).cuda() for i in range(4))].double().cpu().numpy()
    ref = np.array([oracle.wgrad_point(OL, x64, dy64, *map(int, p)) for p in pts])
    assert np.max(np.abs(got - ref)) <= tol * np.max(np.abs(ref)), "dw"

    # dbias = sum of d_conv = sum of dY, every channel
    ref = dy64.reshape(-1, spec.OC).sum(0)
    assert np.max(np.abs(_f64(L.db) - ref)) <= tol * np.max(np.abs(ref)), "dbias"


def _act(kind, t):
    return {0: lambda v: v, 1: torch.relu, 2: torch.tanh, 3: torch.sigmoid}[kind](t)


def _dact(kind, t):
    if kind == 1:
        return (t > 0).double()
    if kind == 2:
        return 1 - torch.tanh(t) ** 2
    if kind == 3:
        s = torch.sigmoid(t)
        return s * (1 - s)
    return torch.ones_like(t)


@pytest.mark.parametrize("name", [c for c in CASES if c != "rl"])
def test_fullsize_batchnorm_properties(name):
    spec, inp = _case(name)
    assert spec.norm == NORM_BATCH
    li = inp["layers"][0]
    rm0 = torch.randn(spec.OC, generator=torch.Generator().manual_seed(5)) * 0.1
    rv0 = torch.rand(spec.OC, generator=torch.Generator().manual_seed(6)) + 0.5
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta, rm0, rv0)
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    L.zero_grad()
    L.fwd_train(x)
    L.bwd(x, dy)
    torch.cuda.synchronize()
    assert abi.conv2d_device_status()[0] == abi.OK
    tol = TOL[spec.dtype]
    C, m = spec.OC, spec.momentum
    u = 2.0 ** -8 if spec.dtype == BF16 else 2.0 ** -24  # storage rounding bound (relative)

    pre = L.pre_act.double().reshape(-1, C)
    mean_g, istd_g = L.save_mean.double(), L.save_inv_std.double()
    var_g = 1.0 / istd_g ** 2 - spec.eps
    # batch statistics: of the conv output before storage rounding, so within the rounding bound of the
    # statistics of the stored values
    mean_s = pre.mean(0)
    var_s = pre.var(0, unbiased=False)
    absmean = pre.abs().mean(0)
    rms = pre.pow(2).mean(0).sqrt()
    std_s = var_s.sqrt()
    assert torch.all((mean_g - mean_s).abs() <= u * absmean + 1e-6 * (mean_s.abs() + std_s)), "batch mean"
    assert torch.all((var_g - var_s).abs() <= 2 * u * std_s * rms + u * u * rms ** 2 + 2e-5 * var_s), "batch var"
    # running statistics: (1 - m) * old + m * batch
    rm_ref = (1 - m) * rm0.double().cuda() + m * mean_g
    rv_ref = (1 - m) * rv0.double().cuda() + m * var_g
    assert torch.all((L.running_mean.double() - rm_ref).abs() <= 1e-6 * (rm_ref.abs() + 1e-3)), "running mean"
    assert torch.all((L.running_var.double() - rv_ref).abs() <= 1e-6 * rv_ref.abs()), "running var"

    g, bt = L.gamma.double(), L.beta.double()
    z = (pre - mean_g) * istd_g
    uact = g * z + bt
    y_ref = _act(spec.act, uact)
    y_err = (L.y.double().reshape(-1, C) - y_ref).abs()
    assert torch.all(y_err <= u * y_ref.abs() + 1e-5 * y_ref.abs().max()), "y"
    del y_ref, y_err

    d = dy.double().reshape(-1, C)
    dn = _dact(spec.act, uact) * d
    dbeta_ref, dgamma_ref = dn.sum(0), (dn * z).sum(0)
    # ReLU inputs within rounding of the kink may take either side on either implementation
    if spec.act == 1:
        near = uact.abs() <= 1e-5 * ((g * z).abs() + bt.abs() + 1e-30)
        slack_b = (near * d.abs()).sum(0)
        slack_g = (near * (d * z).abs()).sum(0)
        del near
    else:
        slack_b = slack_g = torch.zeros_like(dbeta_ref)
    assert torch.all((L.dbeta.double() - dbeta_ref).abs() <= tol * dbeta_ref.abs().max() + slack_b), "dbeta"
    assert torch.all((L.dgamma.double() - dgamma_ref).abs() <= tol * dgamma_ref.abs().max() + slack_g), "dgamma"
    # dbias is analytically zero under training batch norm
    n = pre.shape[0]
    dconv = g * istd_g * (dn - dbeta_ref / n - z * dgamma_ref / n)
    bound = (2e-2 if spec.dtype == BF16 else 1e-4) * dconv.abs().sum(0)
    assert torch.all(L.db.double().abs() <= bound + slack_b * g * istd_g), "dbias"
