"""Conv2dLayer: torch-owned device memory around the C ABI.

PyTorch supplies device memory and the stream; every step of the layer runs
in the library's kernels (through conv2d_layer_gb300.abi). The class holds
the parameters, running statistics, saved forward state and a workspace sized
by conv2d_workspace_size.
"""
import torch

from . import abi

_TORCH_DT = {abi.FP32: torch.float32, abi.BF16: torch.bfloat16}


def _expect(t, name, shape, dtype):
    """The C ABI takes bare pointers and trusts their sizes, so the binding checks each
    caller-supplied tensor before a launch: CUDA memory, dense row-major (NHWC), the
    layer's element type and exactly the shape the descriptor implies. Raises ValueError."""
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} does not match the layer's {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name}: dtype {t.dtype} does not match the layer's {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous (NHWC row-major)")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be in CUDA device memory (got {t.device})")


class Conv2dLayer:
    def __init__(self, spec, w, b=None, gamma=None, beta=None, running_mean=None, running_var=None,
                 device="cuda"):
        self.spec = spec
        self.desc = abi.desc(spec.N, spec.H, spec.W, spec.IC, spec.OC, spec.KH, spec.KW, spec.stride, spec.pad,
                             spec.norm, spec.act, spec.dtype, spec.eps, spec.momentum, spec.bn_eval, spec.groups)
        abi.check(abi.conv2d_validate(self.desc), "conv2d_validate")
        self.dt = _TORCH_DT[spec.dtype]
        dev = torch.device(device)
        f32 = dict(device=dev, dtype=torch.float32)
        self.w = w.to(dev, self.dt).contiguous()
        self.b = (b if b is not None else torch.zeros(spec.OC)).to(**f32).contiguous()
        self.gamma = (gamma if gamma is not None else torch.ones(spec.OC)).to(**f32).contiguous()
        self.beta = (beta if beta is not None else torch.zeros(spec.OC)).to(**f32).contiguous()
        self.running_mean = (running_mean if running_mean is not None else torch.zeros(spec.OC)).to(**f32).clone()
        self.running_var = (running_var if running_var is not None else torch.ones(spec.OC)).to(**f32).clone()
        y_shape = (spec.N, spec.OH, spec.OW, spec.OC)
        self.x_shape = (spec.N, spec.H, spec.W, spec.IC)
        self.y_shape = y_shape
        self.pre_act = torch.empty(y_shape, device=dev, dtype=self.dt)
        self.y = torch.empty(y_shape, device=dev, dtype=self.dt)
        # saved statistics: per channel (batch norm), per image (layer norm) or per image and group
        n_stat = {abi.NORM_LAYER: spec.N, abi.NORM_GROUP: spec.N * spec.groups}.get(spec.norm, spec.OC)
        self.save_mean = torch.zeros(n_stat, **f32)
        self.save_inv_std = torch.zeros(n_stat, **f32)
        self.dw = torch.zeros(spec.OC, spec.KH, spec.KW, spec.IC, **f32)
        self.db = torch.zeros(spec.OC, **f32)
        self.dgamma = torch.zeros(spec.OC, **f32)
        self.dbeta = torch.zeros(spec.OC, **f32)
        self.dx = torch.empty(spec.N, spec.H, spec.W, spec.IC, device=dev, dtype=self.dt)
        ws = max(abi.conv2d_workspace_size(self.desc, op) for op in (0, 1, 2))
        self.ws = torch.empty(max(ws, 256), device=dev, dtype=torch.uint8)

    def zero_grad(self):
        for t in (self.dw, self.db, self.dgamma, self.dbeta):
            t.zero_()

    def fwd_train(self, x, stream=None):
        _expect(x, "x", self.x_shape, self.dt)
        bn = self.spec.norm == abi.NORM_BATCH
        nrm = self.spec.norm != abi.NORM_NONE
        abi.check(abi.conv2d_fwd_train(self.desc, x, self.w, self.b, self.gamma if nrm else None,
                                       self.beta if nrm else None, self.running_mean if bn else None,
                                       self.running_var if bn else None, self.pre_act,
                                       self.save_mean if nrm else None, self.save_inv_std if nrm else None, self.y,
                                       self.ws, stream=stream), "conv2d_fwd_train")
        return self.y

    def fwd_infer(self, x, y=None, stream=None):
        y = self.y if y is None else y
        _expect(x, "x", self.x_shape, self.dt)
        _expect(y, "y", self.y_shape, self.dt)
        abi.check(abi.conv2d_fwd_infer(self.desc, x, self.w, self.b, self.gamma, self.beta, self.running_mean,
                                       self.running_var, y, self.ws, stream=stream), "conv2d_fwd_infer")
        return y

    def bwd(self, x, dy, need_dx=True, need_params=True, stream=None):
        _expect(x, "x", self.x_shape, self.dt)
        _expect(dy, "dy", self.y_shape, self.dt)
        bn = self.spec.norm != abi.NORM_NONE  # batch or layer norm
        abi.check(abi.conv2d_bwd(self.desc, x, self.w, self.gamma if bn else None, self.beta if bn else None,
                                 self.pre_act, self.save_mean if bn else None, self.save_inv_std if bn else None, dy,
                                 self.dx if need_dx else None, self.dw if need_params else None,
                                 self.db if need_params else None,
                                 self.dgamma if (bn and need_params) else None,
                                 self.dbeta if (bn and need_params) else None, self.ws, stream=stream),
                  "conv2d_bwd")
        return self.dx if need_dx else None
