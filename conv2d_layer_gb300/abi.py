"""ctypes binding of libconv2d.so (include/conv2d.h), argument marshalling only.

Every function here has the name of the C entry point it calls and returns its
status code. Tensor arguments are torch CUDA tensors (or None for a NULL
pointer); only their data pointers cross the boundary. `stream` is a
torch.cuda.Stream, a raw cudaStream_t integer, or None for the current torch
stream. Loading fails loudly when the library is missing or cannot be built:
there is no fallback implementation.
"""
import ctypes
import os

from . import build as _build

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT = range(6)
NORM_NONE, NORM_BATCH, NORM_LAYER, NORM_GROUP = 0, 1, 2, 3
ACT_IDENTITY, ACT_RELU, ACT_TANH, ACT_SIGMOID = 0, 1, 2, 3
FP32, BF16 = 0, 1
OP_FWD_TRAIN, OP_FWD_INFER, OP_BWD = 0, 1, 2

EXPORTS = (
    "conv2d_out_hw", "conv2d_validate", "conv2d_workspace_size", "conv2d_fwd_train", "conv2d_fwd_infer",
    "conv2d_bwd", "conv2d_device_status", "conv2d_status_str", "conv2d_prof_enable", "conv2d_prof_read",
    "conv2d_fwd_train_noalloc", "conv2d_selftest_wait_limit",
)


class Conv2dDesc(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("N", "H", "W", "IC", "OC", "KH", "KW", "stride", "pad", "norm", "act",
                                              "dtype")] + [("eps", ctypes.c_float), ("momentum", ctypes.c_float),
                                                           ("bn_eval", ctypes.c_int32), ("groups", ctypes.c_int32)]


class Conv2dError(RuntimeError):
    def __init__(self, status, where=""):
        self.status = status
        super().__init__("%s: %s (%d)" % (where or "conv2d", status_str(status), status))


_lib = None


def lib_path():
    return _build.LIB


def lib():
    """Load (building first if needed) the CUDA library; raises if that is impossible."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if not os.path.exists(path) or os.path.getmtime(path) < _build._deps():
        _build.build()
    L = ctypes.CDLL(path)
    vp, fp, sz, i32 = ctypes.c_void_p, ctypes.POINTER(ctypes.c_float), ctypes.c_size_t, ctypes.c_int
    pd = ctypes.POINTER(Conv2dDesc)
    L.conv2d_out_hw.argtypes = [pd, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    L.conv2d_validate.argtypes = [pd]
    L.conv2d_workspace_size.argtypes = [pd, i32]
    L.conv2d_workspace_size.restype = sz
    L.conv2d_fwd_train.argtypes = [pd] + [vp] * 11 + [vp, sz, vp]
    L.conv2d_fwd_train_noalloc.argtypes = [pd] + [vp] * 11 + [vp]
    L.conv2d_fwd_infer.argtypes = [pd] + [vp] * 8 + [vp, sz, vp]
    L.conv2d_bwd.argtypes = [pd] + [vp] * 13 + [vp, sz, vp]
    L.conv2d_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
    L.conv2d_status_str.argtypes = [i32]
    L.conv2d_status_str.restype = ctypes.c_char_p
    L.conv2d_selftest_wait_limit.argtypes = [vp]
    L.conv2d_prof_enable.argtypes = [i32]
    L.conv2d_prof_read.argtypes = [ctypes.POINTER(ctypes.c_char_p), fp, i32]
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def desc(N, H, W, IC, OC, KH, KW, stride=1, pad=0, norm=NORM_NONE, act=ACT_RELU, dtype=FP32, eps=1e-5,
         momentum=0.1, bn_eval=0, groups=1):
    return Conv2dDesc(N, H, W, IC, OC, KH, KW, stride, pad, norm, act, dtype, eps, momentum, bn_eval, groups)


def status_str(status):
    return lib().conv2d_status_str(int(status)).decode()


def check(status, where=""):
    if status != OK:
        raise Conv2dError(status, where)
    return status


def conv2d_out_hw(d):
    oh, ow = ctypes.c_int32(), ctypes.c_int32()
    rc = lib().conv2d_out_hw(ctypes.byref(d), ctypes.byref(oh), ctypes.byref(ow))
    return rc, oh.value, ow.value


def conv2d_validate(d):
    return lib().conv2d_validate(ctypes.byref(d))


def conv2d_workspace_size(d, op):
    return int(lib().conv2d_workspace_size(ctypes.byref(d), int(op)))


def conv2d_fwd_train(d, x, w, bias, gamma, beta, running_mean, running_var, pre_act, save_mean, save_inv_std, y,
                     ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return lib().conv2d_fwd_train(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(bias), _ptr(gamma), _ptr(beta),
                                  _ptr(running_mean), _ptr(running_var), _ptr(pre_act), _ptr(save_mean),
                                  _ptr(save_inv_std), _ptr(y), _ptr(ws), ws_bytes, _stream(stream))


def conv2d_fwd_train_noalloc(d, x, w, bias, gamma, beta, running_mean, running_var, pre_act, save_mean,
                             save_inv_std, y, stream=None):
    """conv2d_fwd_train with the library's static scratch instead of a caller workspace (no allocation)."""
    return lib().conv2d_fwd_train_noalloc(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(bias), _ptr(gamma), _ptr(beta),
                                          _ptr(running_mean), _ptr(running_var), _ptr(pre_act), _ptr(save_mean),
                                          _ptr(save_inv_std), _ptr(y), _stream(stream))


def conv2d_fwd_infer(d, x, w, bias, gamma, beta, running_mean, running_var, y, ws, ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return lib().conv2d_fwd_infer(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(bias), _ptr(gamma), _ptr(beta),
                                  _ptr(running_mean), _ptr(running_var), _ptr(y), _ptr(ws), ws_bytes,
                                  _stream(stream))


def conv2d_bwd(d, x, w, gamma, beta, pre_act, save_mean, save_inv_std, dy, dx, dw, dbias, dgamma, dbeta, ws,
               ws_bytes=None, stream=None):
    ws_bytes = ws.numel() * ws.element_size() if ws_bytes is None and ws is not None else (ws_bytes or 0)
    return lib().conv2d_bwd(ctypes.byref(d), _ptr(x), _ptr(w), _ptr(gamma), _ptr(beta), _ptr(pre_act),
                            _ptr(save_mean), _ptr(save_inv_std), _ptr(dy), _ptr(dx), _ptr(dw), _ptr(dbias),
                            _ptr(dgamma), _ptr(dbeta), _ptr(ws), ws_bytes, _stream(stream))


def conv2d_device_status(stream=None):
    site = ctypes.c_int32(0)
    rc = lib().conv2d_device_status(_stream(stream), ctypes.byref(site))
    return rc, site.value


def conv2d_selftest_wait_limit(stream=None):
    return lib().conv2d_selftest_wait_limit(_stream(stream))


def conv2d_prof_enable(on):
    return lib().conv2d_prof_enable(1 if on else 0)


def conv2d_prof_read(cap=256):
    names = (ctypes.c_char_p * cap)()
    ms = (ctypes.c_float * cap)()
    n = lib().conv2d_prof_read(names, ms, cap)
    return [(names[i].decode(), ms[i]) for i in range(max(n, 0))]
