"""Pins for the CPU oracle (no GPU): each check fixes the oracle against
something other than itself - finite differences, closed forms, invariants of
batch norm, a hand-worked example, a brute-force restatement of the WGSL
weight-gradient shader, and an independent torch CPU computation.

Formulas pinned: rl-tools page "operations_generic.h" (`forward`, `evaluate`,
`backward_full`); WGSL page "conv2d_backward_weight.wgsl" (per-image dW).
"""
import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand_layer(rng, L, x_scale=1.0):
    x = rng.standard_normal(L.x_shape) * x_scale
    w = rng.standard_normal(L.w_shape) / np.sqrt(L.IC * L.KH * L.KW)
    b = rng.uniform(-0.3, 0.3, L.OC)
    gamma = rng.uniform(0.5, 1.5, L.OC)
    beta = rng.normal(0, 0.1, L.OC)
    dy = rng.standard_normal(L.y_shape)
    return x, w, b, gamma, beta, dy


def _loss(L, x, w, b, gamma, beta, dy):
    out = oracle.fwd_train(L, x, w, b, gamma, beta)
    return float(np.sum(out["y"] * dy))


def _act_inputs(L, x, w, b, gamma, beta):
    out = oracle.fwd_train(L, x, w, b, gamma, beta)
    if L.norm == 0:
        return out["ypre"]
    if L.norm == 2:  # per-sample statistics
        z = (out["ypre"] - out["mean"][:, None, None, None]) * out["inv_std"][:, None, None, None]
    elif L.norm == 3:  # per (image, group) statistics
        z = (out["ypre"] - _group_bcast(L, out["mean"])) * _group_bcast(L, out["inv_std"])
    else:
        z = (out["ypre"] - out["mean"]) * out["inv_std"]
    return gamma * z + beta


def _group_bcast(L, v):
    """[N*G] per-(image, group) values broadcast to [N, 1, 1, OC]."""
    return np.repeat(np.asarray(v).reshape(L.N, L.groups), L.OC // L.groups, axis=1)[:, None, None, :]


def _fd(f, arr, h=1e-5):
    g = np.zeros_like(arr)
    flat, gf = arr.reshape(-1), g.reshape(-1)
    for i in range(flat.size):
        old = flat[i]
        flat[i] = old + h
        fp = f()
        flat[i] = old - h
        fm = f()
        flat[i] = old
        gf[i] = (fp - fm) / (2 * h)
    return g


FD_CASES = [
    # (N,H,W,IC,OC,K,S,P)
    (2, 5, 5, 3, 4, 3, 1, 1),
    (2, 6, 5, 4, 4, 3, 2, 0),
    (1, 9, 9, 3, 4, 3, 4, 1),
    (2, 4, 4, 4, 4, 1, 1, 0),
]


@pytest.mark.parametrize("norm", ["none", "batch", "layer", "group"])
@pytest.mark.parametrize("act", ["identity", "relu", "tanh", "sigmoid"])
@pytest.mark.parametrize("case", FD_CASES)
def test_finite_differences(case, norm, act):
    """Every gradient of L = sum(dY * out) against central differences in double."""
    N, H, W, IC, OC, K, S, P = case
    L = oracle.Layer(N, H, W, IC, OC, K, K, S, P, norm=norm, act=act, groups=2)
    # pick a seed whose activation inputs stay away from the ReLU kink
    for seed in range(50):
        rng = np.random.default_rng(1000 + seed)
        x, w, b, gamma, beta, dy = _rand_layer(rng, L)
        if act != "relu" or np.min(np.abs(_act_inputs(L, x, w, b, gamma, beta))) > 1e-3:
            break
    fwd = oracle.fwd_train(L, x, w, b, gamma, beta)
    g = oracle.bwd(L, x, w, fwd["ypre"], dy, gamma, beta, fwd["mean"], fwd["inv_std"])
    f = lambda: _loss(L, x, w, b, gamma, beta, dy)  # noqa: E731
    checks = [("dx", x, g["dx"]), ("dw", w, g["dw"]), ("db", b, g["db"])]
    if norm != "none":
        checks += [("dgamma", gamma, g["dgamma"]), ("dbeta", beta, g["dbeta"])]
    for name, arr, an in checks:
        num = _fd(f, arr)
        scale = max(np.max(np.abs(num)), np.max(np.abs(an)), 1e-3)
        err = np.max(np.abs(num - an)) / scale
        assert err < 1e-6, (name, err)


def test_one_by_one_kernel_is_a_matmul():
    rng = np.random.default_rng(7)
    L = oracle.Layer(3, 5, 7, 6, 5, 1, 1, 1, 0)
    x, w, b = rng.standard_normal(L.x_shape), rng.standard_normal(L.w_shape), rng.standard_normal(L.OC)
    y = oracle.conv_fwd(L, x, w, b)
    ref = x.reshape(-1, L.IC) @ w.reshape(L.OC, L.IC).T + b
    np.testing.assert_allclose(y.reshape(-1, L.OC), ref, rtol=1e-13, atol=1e-13)


@pytest.mark.parametrize("S", [1, 2, 3])
def test_delta_kernel_is_a_shift(S):
    """W[oc,c,c,ic] = delta(oc,ic), pad c: the conv reproduces X (subsampled by S)."""
    rng = np.random.default_rng(11)
    K, c = 3, 1
    L = oracle.Layer(2, 7, 6, 4, 4, K, K, S, c)
    x = rng.standard_normal(L.x_shape)
    w = np.zeros(L.w_shape)
    for o in range(4):
        w[o, c, c, o] = 1.0
    y = oracle.conv_fwd(L, x, w)
    np.testing.assert_array_equal(y, x[:, ::S, ::S, :][:, :L.OH, :L.OW, :])


def test_shifted_delta_moves_the_image():
    """A delta off the centre shifts the image, with zeros entering at the border."""
    rng = np.random.default_rng(12)
    L = oracle.Layer(1, 5, 5, 2, 2, 3, 3, 1, 1)
    x = rng.standard_normal(L.x_shape)
    w = np.zeros(L.w_shape)
    w[0, 0, 2, 0] = 1.0  # output(oh,ow) = x(oh-1, ow+1)
    w[1, 2, 0, 1] = 1.0  # output(oh,ow) = x(oh+1, ow-1)
    y = oracle.conv_fwd(L, x, w)
    e0 = np.zeros((5, 5))
    e0[1:, :4] = x[0, :4, 1:, 0]
    e1 = np.zeros((5, 5))
    e1[:4, 1:] = x[0, 1:, :4, 1]
    np.testing.assert_array_equal(y[0, :, :, 0], e0)
    np.testing.assert_array_equal(y[0, :, :, 1], e1)


def test_hand_worked_example():
    with open(os.path.join(GOLDEN, "hand_worked_3x3.json")) as f:
        g = json.load(f)
    L = oracle.Layer(1, 3, 3, 1, 1, 2, 2, 1, 0, norm="none", act="identity")
    x = np.array(g["x_hw"], float).reshape(L.x_shape)
    w = np.array(g["w_khkw"], float).reshape(L.w_shape)
    b = np.array([g["bias"]])
    y = oracle.conv_fwd(L, x, w, b)
    np.testing.assert_array_equal(y.reshape(2, 2), np.array(g["ypre_hw"], float))
    mean, var = oracle.bn_batch_stats(L, y)
    assert mean[0] == g["bn_mean"] and var[0] == g["bn_var_biased"]
    out = oracle.bwd(L, x, w, y, np.ones(L.y_shape))
    h = g["dy_all_ones"]
    np.testing.assert_array_equal(out["dx"].reshape(3, 3), np.array(h["identity_none_dx_hw"], float))
    np.testing.assert_array_equal(out["dw"].reshape(2, 2), np.array(h["identity_none_dw_khkw"], float))
    assert out["db"][0] == h["identity_none_dbias"]


def test_batchnorm_invariants():
    rng = np.random.default_rng(5)
    L = oracle.Layer(3, 6, 6, 4, 5, 3, 3, 1, 1, norm="batch", act="tanh", eps=1e-3)
    x, w, b, gamma, beta, dy = _rand_layer(rng, L)
    f = oracle.fwd_train(L, x, w, b, gamma, beta)
    n = L.N * L.OH * L.OW
    z = ((f["ypre"] - f["mean"]) * f["inv_std"]).reshape(n, L.OC)
    mean, var = oracle.bn_batch_stats(L, f["ypre"])
    np.testing.assert_allclose(z.mean(0), 0, atol=1e-12)
    np.testing.assert_allclose((z * z).mean(0), var / (var + L.eps), rtol=1e-12)
    # running statistics after one step from the initial state (0, 1)
    np.testing.assert_allclose(f["running_mean"], L.momentum * mean, rtol=1e-14)
    np.testing.assert_allclose(f["running_var"], (1 - L.momentum) + L.momentum * var, rtol=1e-14)
    # backward: sum of d_conv is 0, its projection on z is the eps leak
    dc, dg, _ = oracle.dconv(L, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    dc = dc.reshape(n, L.OC)
    scale = np.abs(dc).sum(0)
    np.testing.assert_allclose(dc.sum(0) / scale, 0, atol=1e-13)
    leak = f["inv_std"] * gamma * dg * L.eps / (var + L.eps)
    np.testing.assert_allclose((dc * z).sum(0), leak, rtol=1e-9, atol=1e-13 * scale.max())


def test_adjoint_identities():
    """<conv(X), G> = <X, dgrad(G)> and <wgrad(X, G), V> = <conv_V(X), G>."""
    rng = np.random.default_rng(9)
    for (N, H, W, IC, OC, K, S, P) in [(2, 7, 6, 3, 4, 3, 1, 1), (2, 9, 8, 4, 3, 3, 2, 1), (1, 10, 10, 2, 2, 4, 3, 2)]:
        L = oracle.Layer(N, H, W, IC, OC, K, K, S, P)
        x, w = rng.standard_normal(L.x_shape), rng.standard_normal(L.w_shape)
        G, V = rng.standard_normal(L.y_shape), rng.standard_normal(L.w_shape)
        lhs = np.sum(oracle.conv_fwd(L, x, w) * G)
        rhs = np.sum(x * oracle.dgrad(L, G, w))
        assert abs(lhs - rhs) <= 1e-11 * max(1.0, abs(lhs))
        lhs2 = np.sum(oracle.wgrad(L, x, G) * V)
        rhs2 = np.sum(oracle.conv_fwd(L, x, V) * G)
        assert abs(lhs2 - rhs2) <= 1e-11 * max(1.0, abs(lhs2))


def _w1_shader_dw(x_nhwc, dy_nhwc, KH, KW, S, P):
    """The WGSL weight-gradient shader restated: per image, NCHW, one sum per
    weight dW[oc,ic,ky,kx] = sum_{oy,ox} dY[oc,oy,ox] * X[ic, oy*S+ky-P, ox*S+kx-P];
    images summed. Returns [OC,KH,KW,IC] to compare with the oracle."""
    N, H, W, IC = x_nhwc.shape
    _, OH, OW, OC = dy_nhwc.shape
    dw = np.zeros((OC, IC, KH, KW))
    for n in range(N):
        X = np.transpose(x_nhwc[n], (2, 0, 1))
        D = np.transpose(dy_nhwc[n], (2, 0, 1))
        for oc, ic, ky, kx in itertools.product(range(OC), range(IC), range(KH), range(KW)):
            s = 0.0
            for oy in range(OH):
                iy = oy * S + ky
                if iy < P or iy >= H + P:
                    continue
                for ox in range(OW):
                    ix = ox * S + kx
                    if ix < P or ix >= W + P:
                        continue
                    s += D[oc, oy, ox] * X[ic, iy - P, ix - P]
            dw[oc, ic, ky, kx] += s
    return np.transpose(dw, (0, 2, 3, 1))


def test_wgrad_matches_wgsl_shader_math():
    rng = np.random.default_rng(3)
    for (N, H, W, IC, OC, K, S, P) in [(2, 6, 5, 3, 2, 3, 1, 1), (2, 7, 7, 2, 3, 3, 2, 0)]:
        L = oracle.Layer(N, H, W, IC, OC, K, K, S, P)
        x, g = rng.standard_normal(L.x_shape), rng.standard_normal(L.y_shape)
        np.testing.assert_allclose(oracle.wgrad(L, x, g), _w1_shader_dw(x, g, K, K, S, P), rtol=1e-12, atol=1e-12)


def test_gradients_accumulate_and_dx_overwrites():
    rng = np.random.default_rng(4)
    L = oracle.Layer(2, 5, 5, 3, 4, 3, 3, 1, 1, norm="batch", act="relu")
    x, w, b, gamma, beta, dy = _rand_layer(rng, L)
    f = oracle.fwd_train(L, x, w, b, gamma, beta)
    g0 = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    prev = {k: rng.standard_normal(g0[k].shape) for k in ("dw", "db", "dgamma", "dbeta")}
    g1 = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"], **prev)
    for k in prev:
        np.testing.assert_allclose(g1[k], g0[k] + prev[k], rtol=1e-13, atol=1e-13)
    np.testing.assert_array_equal(g1["dx"], g0["dx"])


def test_activation_values():
    v = np.array([-2.0, -0.5, 0.0, 0.5, 2.0])
    np.testing.assert_array_equal(oracle.act("relu", v), [0, 0, 0, 0.5, 2.0])
    np.testing.assert_allclose(oracle.act("tanh", v), np.tanh(v), rtol=1e-15)
    np.testing.assert_allclose(oracle.act("sigmoid", v), 1 / (1 + np.exp(-v)), rtol=1e-15)
    assert oracle.act("sigmoid", 0.0) == 0.5
    np.testing.assert_array_equal(oracle.dact("relu", v), [0, 0, 0, 1, 1])
    h = 1e-6
    for a in ("tanh", "sigmoid", "identity"):
        fd = (oracle.act(a, v + h) - oracle.act(a, v - h)) / (2 * h)
        np.testing.assert_allclose(oracle.dact(a, v), fd, rtol=1e-8, atol=1e-9)


def test_infer_uses_running_statistics():
    rng = np.random.default_rng(8)
    L = oracle.Layer(2, 5, 5, 3, 4, 3, 3, 1, 1, norm="batch", act="sigmoid")
    x, w, b, gamma, beta, _ = _rand_layer(rng, L)
    rm, rv = rng.normal(0, 0.3, L.OC), rng.uniform(0.5, 2.0, L.OC)
    y = oracle.fwd_infer(L, x, w, b, gamma, beta, rm, rv)
    ypre = oracle.conv_fwd(L, x, w, b)
    ref = 1 / (1 + np.exp(-(gamma * (ypre - rm) / np.sqrt(rv + L.eps) + beta)))
    np.testing.assert_allclose(y, ref, rtol=1e-14)
    Ln = oracle.Layer(2, 5, 5, 3, 4, 3, 3, 1, 1, norm="none", act="tanh")
    np.testing.assert_array_equal(oracle.fwd_infer(Ln, x, w, b), oracle.fwd_train(Ln, x, w, b)["y"])


def test_against_torch_cpu_float64():
    """Independent third-party computation (torch CPU, float64, autograd)."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(21)
    acts = {"relu": torch.relu, "tanh": torch.tanh, "sigmoid": torch.sigmoid, "identity": lambda t: t}
    for (N, H, W, IC, OC, K, S, P, norm, act) in [
        (3, 9, 8, 5, 6, 3, 1, 1, "batch", "relu"),
        (2, 11, 11, 4, 8, 5, 2, 2, "batch", "tanh"),
        (2, 10, 9, 3, 4, 4, 3, 0, "none", "sigmoid"),
        (2, 6, 6, 8, 4, 1, 1, 0, "batch", "identity"),
    ]:
        L = oracle.Layer(N, H, W, IC, OC, K, K, S, P, norm=norm, act=act)
        x, w, b, gamma, beta, dy = _rand_layer(rng, L)
        rm0, rv0 = rng.normal(0, 0.2, OC), rng.uniform(0.5, 1.5, OC)
        f = oracle.fwd_train(L, x, w, b, gamma, beta, rm0, rv0)
        g = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])

        tx = torch.tensor(x).permute(0, 3, 1, 2).requires_grad_()
        tw = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_()
        tb = torch.tensor(b).requires_grad_()
        tg = torch.tensor(gamma).requires_grad_()
        tbe = torch.tensor(beta).requires_grad_()
        trm, trv = torch.tensor(rm0), torch.tensor(rv0)
        ypre = F.conv2d(tx, tw, tb, stride=S, padding=P)
        v = F.batch_norm(ypre, trm, trv, tg, tbe, training=True, momentum=L.momentum, eps=L.eps) if norm == "batch" else ypre
        out = acts[act](v)
        tdy = torch.tensor(dy).permute(0, 3, 1, 2)
        (out * tdy).sum().backward()

        nhwc = lambda t: t.detach().permute(0, 2, 3, 1).numpy()  # noqa: E731
        np.testing.assert_allclose(f["ypre"], nhwc(ypre), rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(f["y"], nhwc(out), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dx"], nhwc(tx.grad), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["dw"], tw.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["db"], tb.grad.numpy(), rtol=1e-8, atol=1e-10)
        if norm == "batch":
            n = N * L.OH * L.OW
            np.testing.assert_allclose(g["dgamma"], tg.grad.numpy(), rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(g["dbeta"], tbe.grad.numpy(), rtol=1e-9, atol=1e-11)
            np.testing.assert_allclose(f["running_mean"], trm.numpy(), rtol=1e-12, atol=1e-14)
            # torch keeps the unbiased variance in running_var; the pages keep the biased one
            var_b = (trv.numpy() - (1 - L.momentum) * rv0) / L.momentum * (n - 1) / n
            np.testing.assert_allclose(f["running_var"], (1 - L.momentum) * rv0 + L.momentum * var_b, rtol=1e-12)


def test_store_rounding_matches_bf16_and_fp32_conversion():
    """Pre-activation storage rounding: bf16 round-to-nearest-even (through fp32) and fp32 round-to-nearest,
    checked against torch's conversions and a few hand-picked ties."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(17)
    v = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-30, 30, 4000),
                        [0.0, -0.0, 1.0, 1 + 2 ** -8, 1 + 3 * 2 ** -8, -(1 + 2 ** -8), 65504.0, 3e38, 1e-40]])
    f32 = v.astype(np.float32)
    got = oracle.store_round("bf16", f32.astype(np.float64))
    ref = torch.from_numpy(f32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, ref)
    # ties go to the even mantissa: 1+2^-8 -> 1, 1+3*2^-8 -> 1+2^-6
    assert oracle.store_round("bf16", 1 + 2 ** -8) == 1.0
    assert oracle.store_round("bf16", 1 + 3 * 2 ** -8) == 1 + 2 ** -6
    np.testing.assert_array_equal(oracle.store_round("f32", v), v.astype(np.float32).astype(np.float64))
    np.testing.assert_array_equal(oracle.store_round("f64", v), v)


@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_stored_preactivations_feed_the_statistics(store):
    """With a storage type, Ypre is rounded once; the batch statistics come from the unrounded conv output,
    the normalisation and activation read the rounded value."""
    rng = np.random.default_rng(23)
    L = oracle.Layer(2, 6, 6, 4, 5, 3, 3, 1, 1, norm="batch", act="relu", store=store)
    L0 = oracle.Layer(2, 6, 6, 4, 5, 3, 3, 1, 1, norm="batch", act="relu")
    x, w, b, gamma, beta, _ = _rand_layer(rng, L)
    f = oracle.fwd_train(L, x, w, b, gamma, beta)
    exact = oracle.conv_fwd(L0, x, w, b)
    np.testing.assert_array_equal(f["ypre"], oracle.store_round(store, exact))
    ye = exact.reshape(-1, L.OC)
    np.testing.assert_allclose(f["mean"], ye.mean(0), rtol=1e-13)
    np.testing.assert_allclose(f["inv_std"], 1 / np.sqrt(ye.var(0) + L.eps), rtol=1e-12)
    np.testing.assert_allclose(f["running_var"], 0.9 + 0.1 * ye.var(0), rtol=1e-13)
    z = (f["ypre"] - f["mean"]) * f["inv_std"]
    np.testing.assert_allclose(f["y"], np.maximum(gamma * z + beta, 0), rtol=1e-13, atol=1e-15)


def test_point_functions_match_full_passes():
    """The single-element forms used by the full-size GPU checks agree with the full passes (which the
    adjoint, finite-difference and torch pins fix)."""
    rng = np.random.default_rng(31)
    L = oracle.Layer(2, 9, 8, 3, 5, 3, 3, 2, 1)
    x, w, b = rng.standard_normal(L.x_shape), rng.standard_normal(L.w_shape), rng.standard_normal(L.OC)
    g = rng.standard_normal(L.y_shape)
    y, dx, dw = oracle.conv_fwd(L, x, w, b), oracle.dgrad(L, g, w), oracle.wgrad(L, x, g)
    for n, a, bb, c in [(0, 0, 0, 0), (1, 3, 2, 4), (1, 3, 3, 2)]:
        assert oracle.conv_point(L, x, w, b, n, a, bb, c) == y[n, a, bb, c]
    for n, ih, iw, ic in [(0, 0, 0, 0), (1, 8, 7, 2), (0, 4, 5, 1)]:
        assert abs(oracle.dgrad_point(L, g, w, n, ih, iw, ic) - dx[n, ih, iw, ic]) <= 1e-12
    for oc, kh, kw, ic in [(0, 0, 0, 0), (4, 2, 1, 2)]:
        assert abs(oracle.wgrad_point(L, x, g, oc, kh, kw, ic) - dw[oc, kh, kw, ic]) <= 1e-12


@pytest.mark.parametrize("act", ["relu", "tanh", "sigmoid"])
def test_eval_mode_batchnorm_finite_differences(act):
    """Batch norm in evaluation mode inside training: running statistics, nothing updated; every gradient
    against central differences."""
    L = oracle.Layer(2, 6, 5, 3, 4, 3, 3, 1, 1, norm="batch", act=act, bn_eval=True)
    for seed in range(50):
        rng = np.random.default_rng(2000 + seed)
        x, w, b, gamma, beta, dy = _rand_layer(rng, L)
        rm, rv = rng.normal(0, 0.3, L.OC), rng.uniform(0.5, 2.0, L.OC)
        f = oracle.fwd_train(L, x, w, b, gamma, beta, rm, rv)
        u = gamma * (f["ypre"] - f["mean"]) * f["inv_std"] + beta
        if act != "relu" or np.min(np.abs(u)) > 1e-3:
            break
    np.testing.assert_array_equal(f["running_mean"], rm)
    np.testing.assert_array_equal(f["running_var"], rv)
    np.testing.assert_array_equal(f["mean"], rm)
    np.testing.assert_allclose(f["inv_std"], 1 / np.sqrt(rv + L.eps), rtol=1e-15)
    g = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    loss = lambda: float(np.sum(oracle.fwd_train(L, x, w, b, gamma, beta, rm, rv)["y"] * dy))  # noqa: E731
    for name, arr in (("dx", x), ("dw", w), ("db", b), ("dgamma", gamma), ("dbeta", beta)):
        num = _fd(loss, arr)
        scale = max(np.max(np.abs(num)), 1e-3)
        assert np.max(np.abs(num - g[name])) / scale < 1e-6, name


def test_eval_mode_against_torch_cpu():
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(22)
    L = oracle.Layer(2, 9, 8, 4, 6, 3, 3, 2, 1, norm="batch", act="tanh", bn_eval=True)
    x, w, b, gamma, beta, dy = _rand_layer(rng, L)
    rm, rv = rng.normal(0, 0.3, L.OC), rng.uniform(0.5, 2.0, L.OC)
    f = oracle.fwd_train(L, x, w, b, gamma, beta, rm, rv)
    g = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    tx = torch.tensor(x).permute(0, 3, 1, 2).requires_grad_()
    tw = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_()
    tb, tg, tbe = (torch.tensor(v).requires_grad_() for v in (b, gamma, beta))
    out = torch.tanh(F.batch_norm(F.conv2d(tx, tw, tb, stride=2, padding=1), torch.tensor(rm), torch.tensor(rv),
                                  tg, tbe, training=False, eps=L.eps))
    (out * torch.tensor(dy).permute(0, 3, 1, 2)).sum().backward()
    nhwc = lambda t: t.detach().permute(0, 2, 3, 1).numpy()  # noqa: E731
    np.testing.assert_allclose(f["y"], nhwc(out), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(g["dx"], nhwc(tx.grad), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dw"], tw.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["db"], tb.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dgamma"], tg.grad.numpy(), rtol=1e-9, atol=1e-11)
    np.testing.assert_allclose(g["dbeta"], tbe.grad.numpy(), rtol=1e-9, atol=1e-11)


# ---------------------------------------------------------------- layer norm
def _per_image(a, N):
    return a.reshape(N, -1)


def test_layernorm_invariants():
    """Layer norm (per-sample statistics over OH*OW*OC): z has mean 0 and mean square var/(var+eps) per
    image; the backward's d_conv sums to 0 per image and its projection on z is the eps leak; a common shift
    of every bias leaves the output unchanged, so the bias gradient sums to 0 over channels."""
    rng = np.random.default_rng(41)
    L = oracle.Layer(3, 6, 5, 4, 5, 3, 3, 1, 1, norm="layer", act="tanh", eps=1e-3)
    x, w, b, gamma, beta, dy = _rand_layer(rng, L)
    f = oracle.fwd_train(L, x, w, b, gamma, beta)
    assert f["mean"].shape == (L.N,) and f["inv_std"].shape == (L.N,)
    yp = _per_image(f["ypre"], L.N)
    var = yp.var(1)
    np.testing.assert_allclose(f["mean"], yp.mean(1), rtol=1e-13)
    np.testing.assert_allclose(f["inv_std"], 1 / np.sqrt(var + L.eps), rtol=1e-13)
    z = (yp - f["mean"][:, None]) * f["inv_std"][:, None]
    np.testing.assert_allclose(z.mean(1), 0, atol=1e-13)
    np.testing.assert_allclose((z * z).mean(1), var / (var + L.eps), rtol=1e-12)
    # no running statistics under layer norm
    np.testing.assert_array_equal(f["running_mean"], np.zeros(L.OC))
    np.testing.assert_array_equal(f["running_var"], np.ones(L.OC))
    dc, dg, _ = oracle.dconv(L, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    dc = _per_image(dc, L.N)
    scale = np.abs(dc).sum(1)
    np.testing.assert_allclose(dc.sum(1) / scale, 0, atol=1e-13)
    u = gamma * z.reshape(L.y_shape) + beta
    dzz = _per_image(oracle.dact("tanh", u) * dy * gamma * z.reshape(L.y_shape), L.N).sum(1)
    leak = f["inv_std"] * dzz * L.eps / (var + L.eps)
    np.testing.assert_allclose((dc * z).sum(1), leak, rtol=1e-9, atol=1e-13 * scale.max())
    # bias shift invariance
    f2 = oracle.fwd_train(L, x, w, b + 0.37, gamma, beta)
    np.testing.assert_allclose(f2["y"], f["y"], rtol=1e-12, atol=1e-13)
    g = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    assert abs(g["db"].sum()) <= 1e-12 * np.abs(g["db"]).sum() + 1e-14


def test_layernorm_against_torch_cpu_float64():
    """Independent computation: torch CPU float64 conv2d + layer_norm over (C, H, W) with the per-channel
    gamma / beta broadcast over the image, autograd for every gradient."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(43)
    acts = {"relu": torch.relu, "tanh": torch.tanh, "sigmoid": torch.sigmoid, "identity": lambda t: t}
    for (N, H, W, IC, OC, K, S, P, act) in [
        (3, 9, 8, 5, 6, 3, 1, 1, "relu"),
        (2, 11, 11, 4, 8, 5, 2, 2, "sigmoid"),
        (2, 6, 6, 8, 4, 1, 1, 0, "identity"),
    ]:
        L = oracle.Layer(N, H, W, IC, OC, K, K, S, P, norm="layer", act=act)
        x, w, b, gamma, beta, dy = _rand_layer(rng, L)
        f = oracle.fwd_train(L, x, w, b, gamma, beta)
        g = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
        tx = torch.tensor(x).permute(0, 3, 1, 2).requires_grad_()
        tw = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_()
        tb, tg, tbe = (torch.tensor(v).requires_grad_() for v in (b, gamma, beta))
        ypre = F.conv2d(tx, tw, tb, stride=S, padding=P)
        shp = (OC, L.OH, L.OW)
        v = F.layer_norm(ypre, shp, tg[:, None, None].expand(shp), tbe[:, None, None].expand(shp), eps=L.eps)
        out = acts[act](v)
        (out * torch.tensor(dy).permute(0, 3, 1, 2)).sum().backward()
        nhwc = lambda t: t.detach().permute(0, 2, 3, 1).numpy()  # noqa: E731
        np.testing.assert_allclose(f["y"], nhwc(out), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dx"], nhwc(tx.grad), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["dw"], tw.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["db"], tb.grad.numpy(), rtol=1e-8, atol=1e-10)
        np.testing.assert_allclose(g["dgamma"], tg.grad.numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["dbeta"], tbe.grad.numpy(), rtol=1e-9, atol=1e-11)


@pytest.mark.parametrize("store", ["f32", "bf16"])
def test_layernorm_statistics_come_from_the_stored_values(store):
    """Under layer norm the per-sample statistics are those of the stored pre-activations (the pages'
    LAYER_NORM branch reads `pre_activations`), and inference recomputes the same statistics, so it
    matches the training forward."""
    rng = np.random.default_rng(45)
    L = oracle.Layer(2, 6, 6, 4, 5, 3, 3, 1, 1, norm="layer", act="relu", store=store)
    L0 = oracle.Layer(2, 6, 6, 4, 5, 3, 3, 1, 1, norm="layer", act="relu")
    x, w, b, gamma, beta, _ = _rand_layer(rng, L)
    f = oracle.fwd_train(L, x, w, b, gamma, beta)
    stored = oracle.store_round(store, oracle.conv_fwd(L0, x, w, b))
    np.testing.assert_array_equal(f["ypre"], stored)
    ys = _per_image(stored, L.N)
    np.testing.assert_allclose(f["mean"], ys.mean(1), rtol=1e-13)
    np.testing.assert_allclose(f["inv_std"], 1 / np.sqrt(ys.var(1) + L.eps), rtol=1e-12)
    z = (ys - f["mean"][:, None]) * f["inv_std"][:, None]
    np.testing.assert_allclose(f["y"], np.maximum(gamma * z.reshape(L.y_shape) + beta, 0), rtol=1e-13,
                               atol=1e-15)
    np.testing.assert_allclose(oracle.fwd_infer(L, x, w, b, gamma, beta), f["y"], rtol=1e-14, atol=1e-15)


# ---------------------------------------------------------------- group norm
def test_groupnorm_with_one_group_is_layer_norm():
    """Group norm with a single group normalises over the whole image: the layer-norm code path."""
    rng = np.random.default_rng(51)
    for store in (None, "bf16"):
        Lg = oracle.Layer(2, 7, 6, 3, 6, 3, 3, 1, 1, norm="group", act="sigmoid", groups=1, store=store)
        Ll = oracle.Layer(2, 7, 6, 3, 6, 3, 3, 1, 1, norm="layer", act="sigmoid", store=store)
        x, w, b, gamma, beta, dy = _rand_layer(rng, Lg)
        fg, fl = oracle.fwd_train(Lg, x, w, b, gamma, beta), oracle.fwd_train(Ll, x, w, b, gamma, beta)
        for k in ("ypre", "y", "mean", "inv_std"):
            np.testing.assert_allclose(fg[k], fl[k], rtol=1e-13, atol=1e-15)
        gg = oracle.bwd(Lg, x, w, fg["ypre"], dy, gamma, beta, fg["mean"], fg["inv_std"])
        gl = oracle.bwd(Ll, x, w, fl["ypre"], dy, gamma, beta, fl["mean"], fl["inv_std"])
        for k in ("dx", "dw", "db", "dgamma", "dbeta"):
            np.testing.assert_allclose(gg[k], gl[k], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(oracle.fwd_infer(Lg, x, w, b, gamma, beta),
                                   oracle.fwd_infer(Ll, x, w, b, gamma, beta), rtol=1e-13, atol=1e-15)


def test_groupnorm_against_torch_cpu_float64():
    """Independent computation: torch CPU float64 conv2d + group_norm (and, with one channel per group,
    instance norm), autograd for every gradient."""
    torch = pytest.importorskip("torch")
    F = torch.nn.functional
    rng = np.random.default_rng(53)
    acts = {"relu": torch.relu, "tanh": torch.tanh, "sigmoid": torch.sigmoid, "identity": lambda t: t}
    for (N, H, W, IC, OC, K, S, P, G, act) in [
        (3, 9, 8, 5, 8, 3, 1, 1, 2, "relu"),
        (2, 11, 11, 4, 12, 5, 2, 2, 3, "tanh"),
        (2, 6, 6, 8, 6, 1, 1, 0, 6, "identity"),
    ]:
        L = oracle.Layer(N, H, W, IC, OC, K, K, S, P, norm="group", act=act, groups=G)
        x, w, b, gamma, beta, dy = _rand_layer(rng, L)
        f = oracle.fwd_train(L, x, w, b, gamma, beta)
        g = oracle.bwd(L, x, w, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
        tx = torch.tensor(x).permute(0, 3, 1, 2).requires_grad_()
        tw = torch.tensor(w).permute(0, 3, 1, 2).contiguous().requires_grad_()
        tb, tg, tbe = (torch.tensor(v).requires_grad_() for v in (b, gamma, beta))
        v = F.group_norm(F.conv2d(tx, tw, tb, stride=S, padding=P), G, tg, tbe, eps=L.eps)
        if G == OC:
            vi = F.instance_norm(F.conv2d(tx, tw, tb, stride=S, padding=P), weight=tg, bias=tbe, eps=L.eps)
            np.testing.assert_allclose(v.detach().numpy(), vi.detach().numpy(), rtol=1e-12, atol=1e-13)
        out = acts[act](v)
        (out * torch.tensor(dy).permute(0, 3, 1, 2)).sum().backward()
        nhwc = lambda t: t.detach().permute(0, 2, 3, 1).numpy()  # noqa: E731
        np.testing.assert_allclose(f["y"], nhwc(out), rtol=1e-10, atol=1e-12)
        np.testing.assert_allclose(g["dx"], nhwc(tx.grad), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["dw"], tw.grad.permute(0, 2, 3, 1).numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["db"], tb.grad.numpy(), rtol=1e-8, atol=1e-10)
        np.testing.assert_allclose(g["dgamma"], tg.grad.numpy(), rtol=1e-9, atol=1e-11)
        np.testing.assert_allclose(g["dbeta"], tbe.grad.numpy(), rtol=1e-9, atol=1e-11)


def test_groupnorm_invariants_and_stored_statistics():
    """Per (image, group): statistics of the stored values, z of mean 0, d_conv summing to 0; inference
    recomputes the same statistics."""
    rng = np.random.default_rng(55)
    L = oracle.Layer(2, 6, 6, 4, 8, 3, 3, 1, 1, norm="group", act="tanh", groups=4, store="bf16")
    L0 = oracle.Layer(2, 6, 6, 4, 8, 3, 3, 1, 1, norm="group", act="tanh", groups=4)
    x, w, b, gamma, beta, dy = _rand_layer(rng, L)
    f = oracle.fwd_train(L, x, w, b, gamma, beta)
    assert f["mean"].shape == (L.N * L.groups,)
    stored = oracle.store_round("bf16", oracle.conv_fwd(L0, x, w, b))
    np.testing.assert_array_equal(f["ypre"], stored)
    cpg = L.OC // L.groups
    grp = stored.reshape(L.N, -1, L.groups, cpg).transpose(0, 2, 1, 3).reshape(L.N * L.groups, -1)
    np.testing.assert_allclose(f["mean"], grp.mean(1), rtol=1e-13)
    np.testing.assert_allclose(f["inv_std"], 1 / np.sqrt(grp.var(1) + L.eps), rtol=1e-12)
    dc, _, _ = oracle.dconv(L, f["ypre"], dy, gamma, beta, f["mean"], f["inv_std"])
    dg = dc.reshape(L.N, -1, L.groups, cpg).transpose(0, 2, 1, 3).reshape(L.N * L.groups, -1)
    np.testing.assert_allclose(dg.sum(1) / np.abs(dg).sum(1), 0, atol=1e-13)
    np.testing.assert_allclose(oracle.fwd_infer(L, x, w, b, gamma, beta), f["y"], rtol=1e-14, atol=1e-15)
