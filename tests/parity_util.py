"""Helpers for the GPU parity tests: run one layer through the C ABI and the
same seeded inputs through the CPU oracle, and compare per output tensor.

Tolerance (per output tensor): max|gpu - ref| / max|ref| <= 1e-5 for the FP32
(3xTF32) mode and <= 2e-2 for the BF16 mode; running statistics <= 1e-5.
dBias under training batch norm (and under group norm with one channel per
group) is analytically zero, so it is checked against the scale of the summed
terms instead: |dbias[c]| <= t * sum|d_conv[:,c]| with t = 1e-4 (FP32) / 2e-2
(BF16). Under layer norm the saved statistics are
per image ([N]) and are compared like the other outputs.
"""
import numpy as np
import torch

import oracle
from conv2d_layer_gb300 import abi
from conv2d_layer_gb300.layer import Conv2dLayer
from conv2d_layer_gb300.workloads import BF16, NORM_BATCH, NORM_GROUP, NORM_NONE

TOL = {0: 1e-5, 1: 2e-2}
STAT_TOL = 1e-5
DBIAS_TOL = {0: 1e-4, 1: 2e-2}


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def rel_err(a, ref):
    a, ref = np.asarray(a, np.float64), np.asarray(ref, np.float64)
    scale = np.max(np.abs(ref))
    return float(np.max(np.abs(a - ref)) / (scale if scale > 0 else 1.0))


def oracle_layer(spec):
    """Oracle layer with the pre-activations stored in the layer's element type, as the pages do."""
    return oracle.Layer(spec.N, spec.H, spec.W, spec.IC, spec.OC, spec.KH, spec.KW, spec.stride, spec.pad,
                        norm=spec.norm, act=spec.act, eps=spec.eps, momentum=spec.momentum,
                        store="bf16" if spec.dtype == BF16 else "f32", bn_eval=spec.bn_eval,
                        groups=spec.groups)


def run_pair(spec, inp, prev_grads=False, need_dx=True, need_params=True, seed=0):
    """Training forward + backward on the GPU and in the oracle. Returns (gpu, ref) dicts of float64 arrays."""
    li = inp["layers"][0]
    x, dy = inp["x"], inp["dy"]
    L = Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta, li.running_mean, li.running_var)
    xg, dyg = x.cuda(), dy.cuda()
    rng = np.random.default_rng(seed)
    prev = None
    if prev_grads:
        prev = {k: rng.standard_normal(s).astype(np.float32).astype(np.float64) for k, s in
                (("dw", tuple(L.dw.shape)), ("db", (spec.OC,)), ("dgamma", (spec.OC,)), ("dbeta", (spec.OC,)))}
        for k, t in (("dw", L.dw), ("db", L.db), ("dgamma", L.dgamma), ("dbeta", L.dbeta)):
            t.copy_(torch.from_numpy(prev[k]).float())
    else:
        L.zero_grad()
    L.fwd_train(xg)
    L.bwd(xg, dyg, need_dx=need_dx, need_params=need_params)
    torch.cuda.synchronize()
    st = abi.conv2d_device_status()
    assert st[0] == abi.OK, st
    gpu = dict(ypre=f64(L.pre_act), y=f64(L.y), mean=f64(L.save_mean), inv_std=f64(L.save_inv_std),
               running_mean=f64(L.running_mean), running_var=f64(L.running_var), dx=f64(L.dx), dw=f64(L.dw),
               db=f64(L.db), dgamma=f64(L.dgamma), dbeta=f64(L.dbeta))

    OL = oracle_layer(spec)
    xd, wd = f64(x), f64(li.w)
    f = oracle.fwd_train(OL, xd, wd, f64(li.b), f64(li.gamma), f64(li.beta), f64(li.running_mean),
                         f64(li.running_var))
    kw = {}
    if prev is not None:
        kw = dict(dw=prev["dw"], db=prev["db"], dgamma=prev["dgamma"], dbeta=prev["dbeta"])
    g = oracle.bwd(OL, xd, wd, f["ypre"], f64(dy), f64(li.gamma), f64(li.beta), f["mean"], f["inv_std"],
                   need_dx=need_dx, need_params=need_params, **kw)
    ref = dict(f)
    ref.update(g)
    if prev is not None:
        ref["prev"] = prev
    return gpu, ref


def check_pair(spec, gpu, ref, need_dx=True, need_params=True):
    """Assert the parity bar; returns the per-tensor errors for reporting."""
    tol = TOL[spec.dtype]
    errs = {}
    names = ["ypre", "y"]
    if spec.norm != NORM_NONE:
        names += ["mean", "inv_std"]
    if need_dx:
        names += ["dx"]
    # dbias is analytically zero under training batch norm and under group norm with one channel per
    # group (instance norm): a shift of a channel's bias leaves the output unchanged
    bn_train = (spec.norm == NORM_BATCH and not spec.bn_eval) or (spec.norm == NORM_GROUP and spec.groups == spec.OC)
    if need_params:
        names += ["dw"]
        if spec.norm != NORM_NONE:
            names += ["dgamma", "dbeta"]
        if not bn_train:
            names += ["db"]
    for k in names:
        errs[k] = rel_err(gpu[k], ref[k])
    bad = {k: v for k, v in errs.items() if not v <= tol}
    if spec.norm == NORM_BATCH:
        for k in ("running_mean", "running_var"):
            errs[k] = rel_err(gpu[k], ref[k])
            if not errs[k] <= STAT_TOL:
                bad[k] = errs[k]
    if spec.norm != NORM_NONE:
        if need_params and bn_train:
            dc = ref["dconv"].reshape(-1, spec.OC)
            bound = DBIAS_TOL[spec.dtype] * np.abs(dc).sum(0)
            prev = ref["prev"]["db"] if "prev" in ref else 0.0
            dev = np.abs(gpu["db"] - prev)
            errs["db_vs_scale"] = float(np.max(dev / np.maximum(bound, 1e-30)))
            if not np.all(dev <= bound):
                bad["db"] = errs["db_vs_scale"]
    assert not bad, "parity failed (tol %g): %s; all: %s" % (tol, bad, errs)
    return errs
