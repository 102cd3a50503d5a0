"""CPU oracle for the conv2d training step (numpy float64 in, float64 out).

TEST INFRASTRUCTURE ONLY: imported by tests/, by the smoke check and by the
benchmark's CPU-baseline leg, never by the product library. It shares no code
with the CUDA path; the two meet only through the seeded inputs of
``conv2d_layer_gb300.workloads``.

Every function forwards to ``conv2d_oracle.c`` (plain nested loops in double,
two-pass batch statistics), which restates the rl-tools page
"operations_generic.h" (`forward`, `evaluate`, `backward_full`); the C file's
header lists the readings taken where the page is silent.

Pinned by tests/test_oracle_pins.py (finite differences, closed forms,
invariants, a brute-force restatement of the WGSL weight-gradient shader and
an independent torch CPU computation). No function here is "parity unpinned".
"""
import ctypes
import numpy as np

from . import build as _build

ACT = {"identity": 0, "relu": 1, "tanh": 2, "sigmoid": 3}
STORE = {None: 0, "f64": 0, "f32": 1, "bf16": 2}
NORM = {"none": 0, "batch": 1, "layer": 2, "group": 3}


class _Desc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("N", "H", "W", "IC", "OC", "KH", "KW", "S", "P", "norm", "act",
                                              "store", "bn_eval", "groups")] + [
        ("eps", ctypes.c_double),
        ("momentum", ctypes.c_double),
    ]


_lib = None


def _load():
    global _lib
    if _lib is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        dp = ctypes.POINTER(ctypes.c_double)
        pd = ctypes.POINTER(_Desc)
        lib.oracle_conv_point.restype = ctypes.c_double
        lib.oracle_conv_point.argtypes = [pd, dp, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_dgrad_point.restype = ctypes.c_double
        lib.oracle_dgrad_point.argtypes = [pd, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_wgrad_point.restype = ctypes.c_double
        lib.oracle_wgrad_point.argtypes = [pd, dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int]
        lib.oracle_act.restype = ctypes.c_double
        lib.oracle_act.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.oracle_dact.restype = ctypes.c_double
        lib.oracle_dact.argtypes = [ctypes.c_int, ctypes.c_double]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_store_round.restype = ctypes.c_double
        lib.oracle_store_round.argtypes = [ctypes.c_int, ctypes.c_double]
        _lib = lib
    return _lib


def num_threads() -> int:
    return int(_load().oracle_num_threads())


class Layer:
    """Layer spec: N,H,W,IC,OC,KH,KW,stride,pad, normalization, activation, eps, momentum, and the
    element type the pre-activations are stored in (store: None/"f64" keeps fp64, "f32", "bf16")."""

    def __init__(self, N, H, W, IC, OC, KH, KW, stride=1, pad=0, norm="none", act="identity",
                 eps=1e-5, momentum=0.1, store=None, bn_eval=False, groups=1):
        self.N, self.H, self.W, self.IC, self.OC = N, H, W, IC, OC
        self.KH, self.KW, self.S, self.P = KH, KW, stride, pad
        self.norm = norm if isinstance(norm, int) else NORM[norm]
        self.act = act if isinstance(act, int) else ACT[act]
        self.eps, self.momentum = float(eps), float(momentum)
        self.store = store if isinstance(store, int) else STORE[store]
        self.bn_eval = 1 if bn_eval else 0
        self.groups = int(groups)  # group norm: channel groups (dividing OC)
        self.OH = (H + 2 * pad - KH) // stride + 1
        self.OW = (W + 2 * pad - KW) // stride + 1

    @property
    def n_stats(self):
        """Entries of the saved mean / inv_std."""
        return {2: self.N, 3: self.N * self.groups}.get(self.norm, self.OC)

    def _c(self):
        return _Desc(self.N, self.H, self.W, self.IC, self.OC, self.KH, self.KW, self.S, self.P,
                     self.norm, self.act, self.store, self.bn_eval, self.groups, self.eps, self.momentum)

    @property
    def x_shape(self):
        return (self.N, self.H, self.W, self.IC)

    @property
    def w_shape(self):
        return (self.OC, self.KH, self.KW, self.IC)

    @property
    def y_shape(self):
        return (self.N, self.OH, self.OW, self.OC)


def _d(a, shape=None):
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None:
        a = a.reshape(shape)
    return a


def _p(a):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _zeros_if_none(a, n):
    return np.zeros(n) if a is None else _d(a).reshape(n).copy()


def conv_fwd(L: Layer, x, w, b=None):
    """Ypre = conv(X, W) + b (NHWC), float64."""
    lib = _load()
    x, w = _d(x, L.x_shape), _d(w, L.w_shape)
    b = _zeros_if_none(b, L.OC)
    y = np.empty(L.y_shape)
    c = L._c()
    lib.oracle_conv_fwd(ctypes.byref(c), _p(x), _p(w), _p(b), _p(y))
    return y


def conv_point(L: Layer, x, w, b, n, oh, ow, oc):
    lib = _load()
    c = L._c()
    return lib.oracle_conv_point(ctypes.byref(c), _p(x), _p(w), _p(b), n, oh, ow, oc)


def bn_batch_stats(L: Layer, ypre):
    lib = _load()
    ypre = _d(ypre, L.y_shape)
    mean, var = np.empty(L.OC), np.empty(L.OC)
    c = L._c()
    lib.oracle_bn_batch_stats(ctypes.byref(c), _p(ypre), _p(mean), _p(var))
    return mean, var


def fwd_train(L: Layer, x, w, b, gamma=None, beta=None, running_mean=None, running_var=None):
    """Training forward. Returns dict(ypre, mean, inv_std, y, running_mean, running_var)."""
    lib = _load()
    x, w = _d(x, L.x_shape), _d(w, L.w_shape)
    b = _zeros_if_none(b, L.OC)
    gamma = _zeros_if_none(gamma, L.OC) if gamma is not None else np.ones(L.OC)
    beta = _zeros_if_none(beta, L.OC)
    rm = _zeros_if_none(running_mean, L.OC)
    rv = np.ones(L.OC) if running_var is None else _d(running_var).reshape(L.OC).copy()
    ypre, y = np.empty(L.y_shape), np.empty(L.y_shape)
    ns = L.n_stats  # per channel (batch norm), per image (layer norm), per (image, group) (group norm)
    mean, inv_std = np.zeros(max(ns, L.OC)), np.zeros(max(ns, L.OC))
    c = L._c()
    lib.oracle_fwd_train(ctypes.byref(c), _p(x), _p(w), _p(b), _p(gamma), _p(beta), _p(rm), _p(rv),
                         _p(ypre), _p(mean), _p(inv_std), _p(y))
    return dict(ypre=ypre, mean=mean[:ns], inv_std=inv_std[:ns], y=y, running_mean=rm, running_var=rv)


def fwd_infer(L: Layer, x, w, b, gamma=None, beta=None, running_mean=None, running_var=None):
    lib = _load()
    x, w = _d(x, L.x_shape), _d(w, L.w_shape)
    b = _zeros_if_none(b, L.OC)
    gamma = _d(gamma).reshape(L.OC) if gamma is not None else np.ones(L.OC)
    beta = _zeros_if_none(beta, L.OC)
    rm = _zeros_if_none(running_mean, L.OC)
    rv = np.ones(L.OC) if running_var is None else _d(running_var).reshape(L.OC)
    y = np.empty(L.y_shape)
    c = L._c()
    lib.oracle_fwd_infer(ctypes.byref(c), _p(x), _p(w), _p(b), _p(gamma), _p(beta), _p(rm), _p(rv), _p(y))
    return y


def dconv(L: Layer, ypre, dy, gamma=None, beta=None, mean=None, inv_std=None):
    """Gradient at the conv output, plus (BN) the dgamma / dbeta sums. Returns (dconv, dgamma, dbeta)."""
    lib = _load()
    ypre, dy = _d(ypre, L.y_shape), _d(dy, L.y_shape)
    gamma = _d(gamma).reshape(L.OC) if gamma is not None else np.ones(L.OC)
    beta = _zeros_if_none(beta, L.OC)
    ns = L.n_stats
    mean = _zeros_if_none(mean, ns)
    inv_std = _d(inv_std).reshape(ns) if inv_std is not None else np.ones(ns)
    out = np.empty(L.y_shape)
    dg, dbt = np.zeros(L.OC), np.zeros(L.OC)
    c = L._c()
    lib.oracle_dconv(ctypes.byref(c), _p(gamma), _p(beta), _p(ypre), _p(mean), _p(inv_std), _p(dy), _p(out),
                     _p(dg), _p(dbt))
    return out, dg, dbt


def dgrad(L: Layer, dconv_, w):
    lib = _load()
    dc, w = _d(dconv_, L.y_shape), _d(w, L.w_shape)
    dx = np.empty(L.x_shape)
    c = L._c()
    lib.oracle_dgrad(ctypes.byref(c), _p(dc), _p(w), _p(dx))
    return dx


def wgrad(L: Layer, x, dconv_):
    lib = _load()
    x, dc = _d(x, L.x_shape), _d(dconv_, L.y_shape)
    dw = np.zeros(L.w_shape)
    c = L._c()
    lib.oracle_wgrad(ctypes.byref(c), _p(x), _p(dc), _p(dw))
    return dw


def dgrad_point(L: Layer, dconv_, w, n, ih, iw, ic):
    lib = _load()
    c = L._c()
    return lib.oracle_dgrad_point(ctypes.byref(c), _p(dconv_), _p(w), n, ih, iw, ic)


def wgrad_point(L: Layer, x, dconv_, oc, kh, kw, ic):
    lib = _load()
    c = L._c()
    return lib.oracle_wgrad_point(ctypes.byref(c), _p(x), _p(dconv_), oc, kh, kw, ic)


def bwd(L: Layer, x, w, ypre, dy, gamma=None, beta=None, mean=None, inv_std=None, need_dx=True,
        need_params=True, dw=None, db=None, dgamma=None, dbeta=None):
    """Full backward. Param grads accumulate into the given (or zero) arrays; dx is overwritten.

    Returns dict(dx, dw, db, dgamma, dbeta, dconv)."""
    lib = _load()
    x, w = _d(x, L.x_shape), _d(w, L.w_shape)
    ypre, dy = _d(ypre, L.y_shape), _d(dy, L.y_shape)
    gamma = _d(gamma).reshape(L.OC) if gamma is not None else np.ones(L.OC)
    beta = _zeros_if_none(beta, L.OC)
    ns = L.n_stats
    mean = _zeros_if_none(mean, ns)
    inv_std = _d(inv_std).reshape(ns) if inv_std is not None else np.ones(ns)
    dx = np.empty(L.x_shape) if need_dx else None
    dw = (np.zeros(L.w_shape) if dw is None else _d(dw, L.w_shape).copy()) if need_params else None
    db = _zeros_if_none(db, L.OC) if need_params else None
    dg = _zeros_if_none(dgamma, L.OC) if need_params else None
    dbt = _zeros_if_none(dbeta, L.OC) if need_params else None
    dc = np.empty(L.y_shape)
    c = L._c()
    lib.oracle_bwd(ctypes.byref(c), _p(x), _p(w), _p(gamma), _p(beta), _p(ypre), _p(mean), _p(inv_std), _p(dy),
                   _p(dx), _p(dw), _p(db), _p(dg), _p(dbt), _p(dc))
    return dict(dx=dx, dw=dw, db=db, dgamma=dg, dbeta=dbt, dconv=dc)


def store_round(store, v):
    """Round to the pre-activation storage type (vectorised over an array)."""
    lib = _load()
    k = store if isinstance(store, int) else STORE[store]
    return np.vectorize(lambda t: lib.oracle_store_round(k, float(t)))(v)


def act(kind, v):
    lib = _load()
    k = kind if isinstance(kind, int) else ACT[kind]
    return np.vectorize(lambda t: lib.oracle_act(k, float(t)))(v)


def dact(kind, v):
    lib = _load()
    k = kind if isinstance(kind, int) else ACT[kind]
    return np.vectorize(lambda t: lib.oracle_dact(k, float(t)))(v)
