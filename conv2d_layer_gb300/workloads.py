"""Seeded synthetic inputs for the conv2d training step.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes, distributions and draw order of the five workloads (tiny,
RL encoder, BN layer, mixed two-layer stack, large), so that the oracle and
the CUDA path see identical data. Everything is drawn on the CPU from one
``torch.Generator`` per workload, in fp32, and rounded to bf16
(round-to-nearest-even, ``Tensor.to(torch.bfloat16)``) for the BF16
workloads before either side sees it.

Distributions (second argument of N(.,.) is the standard deviation):
  tiny   X~N(0,1), W~N(0,1/sqrt(27)), b~U(+-1/sqrt(27)), dY~N(0,1)
  rl     X~U(0,1), W~N(0,sqrt(2/256)), b~U(+-1/16), dY~N(0,1)
  bn     X~N(0,1), W~N(0,sqrt(2/576)), b~U(+-1/24), gamma~U(0.5,1.5),
         beta~N(0,0.1), dY~N(0,1)
  mixed  as bn per layer (W std sqrt(2/fan_in), b~U(+-1/sqrt(fan_in))),
         bf16, layer 1 output feeds layer 2
  large  X~N(0,1), W~N(0,sqrt(2/2304)), b~U(+-1/48), gamma/beta as bn,
         dY~N(0,1e-2)
Draw order: X, W, b, gamma, beta, dY, then layer 2's W, b, gamma, beta.
"""
from dataclasses import dataclass, field, replace
import math

import torch

FP32, BF16 = 0, 1
NORM_NONE, NORM_BATCH, NORM_LAYER, NORM_GROUP = 0, 1, 2, 3
ACT_IDENTITY, ACT_RELU, ACT_TANH, ACT_SIGMOID = 0, 1, 2, 3


@dataclass(frozen=True)
class LayerSpec:
    N: int
    H: int
    W: int
    IC: int
    OC: int
    KH: int
    KW: int
    stride: int = 1
    pad: int = 0
    norm: int = NORM_NONE
    act: int = ACT_RELU
    dtype: int = FP32
    eps: float = 1e-5
    momentum: float = 0.1
    bn_eval: int = 0      # batch norm in evaluation mode inside training
    groups: int = 1       # group norm: channel groups

    @property
    def OH(self):
        return (self.H + 2 * self.pad - self.KH) // self.stride + 1

    @property
    def OW(self):
        return (self.W + 2 * self.pad - self.KW) // self.stride + 1

    @property
    def n_pix(self):
        return self.N * self.OH * self.OW

    @property
    def fan_in(self):
        return self.IC * self.KH * self.KW

    def flops_fwd(self):
        """Full-tap convention: 2 * n_pix * OC * KH * KW * IC."""
        return 2.0 * self.n_pix * self.OC * self.KH * self.KW * self.IC

    def flops_step(self):
        return 3.0 * self.flops_fwd()


@dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    layers: tuple
    x_dist: str = "normal"          # "normal" N(0,1) or "uniform" U(0,1)
    w_std: tuple = ()               # per layer
    b_bound: tuple = ()             # per layer
    dy_std: float = 1.0
    bn_params: bool = False


def _spec(**kw):
    return LayerSpec(**kw)


WORKLOADS = {
    "tiny": Workload(
        "tiny", 0,
        (_spec(N=2, H=8, W=8, IC=3, OC=4, KH=3, KW=3, stride=1, pad=1, act=ACT_RELU, dtype=FP32),),
        w_std=(1 / math.sqrt(27),), b_bound=(1 / math.sqrt(27),)),
    "rl": Workload(
        "rl", 1,
        (_spec(N=256, H=84, W=84, IC=4, OC=32, KH=8, KW=8, stride=4, pad=0, act=ACT_RELU, dtype=FP32),),
        x_dist="uniform", w_std=(math.sqrt(2 / 256),), b_bound=(1 / 16,)),
    "bn": Workload(
        "bn", 2,
        (_spec(N=128, H=32, W=32, IC=64, OC=64, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_RELU,
               dtype=FP32),),
        w_std=(math.sqrt(2 / 576),), b_bound=(1 / 24,), bn_params=True),
    "mixed": Workload(
        "mixed", 3,
        (_spec(N=64, H=56, W=56, IC=128, OC=256, KH=1, KW=1, stride=1, pad=0, norm=NORM_BATCH, act=ACT_TANH,
               dtype=BF16),
         _spec(N=64, H=56, W=56, IC=256, OC=256, KH=3, KW=3, stride=2, pad=1, norm=NORM_BATCH, act=ACT_TANH,
               dtype=BF16)),
        w_std=(math.sqrt(2 / 128), math.sqrt(2 / 2304)), b_bound=(1 / math.sqrt(128), 1 / math.sqrt(2304)),
        bn_params=True),
    "large": Workload(
        "large", 4,
        (_spec(N=256, H=56, W=56, IC=256, OC=256, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH, act=ACT_RELU,
               dtype=BF16),),
        w_std=(math.sqrt(2 / 2304),), b_bound=(1 / 48,), dy_std=1e-2, bn_params=True),
}


def _round(t, dtype):
    """Storage rounding of an operand tensor: bf16 (RNE) for BF16 layers, else fp32."""
    if dtype == BF16:
        return t.to(torch.bfloat16)
    return t.contiguous()


@dataclass
class LayerInputs:
    spec: LayerSpec
    w: torch.Tensor           # [OC,KH,KW,IC], operand dtype
    b: torch.Tensor           # [OC] fp32
    gamma: torch.Tensor       # [OC] fp32
    beta: torch.Tensor        # [OC] fp32
    running_mean: torch.Tensor = field(default=None)
    running_var: torch.Tensor = field(default=None)


def _layer_params(g, spec, w_std, b_bound, bn_params):
    w = torch.randn(spec.OC, spec.KH, spec.KW, spec.IC, generator=g) * w_std
    b = (torch.rand(spec.OC, generator=g) * 2 - 1) * b_bound
    if bn_params:
        gamma = torch.rand(spec.OC, generator=g) + 0.5
        beta = torch.randn(spec.OC, generator=g) * 0.1
    else:
        gamma = torch.ones(spec.OC)
        beta = torch.zeros(spec.OC)
    return LayerInputs(spec, _round(w, spec.dtype), b.float(), gamma.float(), beta.float(),
                       torch.zeros(spec.OC), torch.ones(spec.OC))


def make_inputs(name, n_images=None, seed=None, layers=None):
    """Draw the inputs of a workload on the CPU.

    n_images, if given, replaces N of every layer (a bounded sample of the same
    workload: same per-image shapes and distributions). layers, if given,
    replaces the layer specs (used for scaled-down parity cases).
    Returns dict(x, dy, layers=[LayerInputs...]).
    """
    wl = WORKLOADS[name]
    specs = list(layers if layers is not None else wl.layers)
    if n_images is not None:
        specs = [replace(s, N=n_images) for s in specs]
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    s0 = specs[0]
    if wl.x_dist == "uniform":
        x = torch.rand(s0.N, s0.H, s0.W, s0.IC, generator=g)
    else:
        x = torch.randn(s0.N, s0.H, s0.W, s0.IC, generator=g)
    x = _round(x, s0.dtype)
    params = [_layer_params(g, specs[0], wl.w_std[0], wl.b_bound[0], wl.bn_params)]
    sl = specs[-1]
    dy = _round(torch.randn(sl.N, sl.OH, sl.OW, sl.OC, generator=g) * wl.dy_std, sl.dtype)
    for i in range(1, len(specs)):
        params.append(_layer_params(g, specs[i], wl.w_std[i], wl.b_bound[i], wl.bn_params))
    return dict(x=x, dy=dy, layers=params)


def random_layer_inputs(spec, seed, x_dist="normal", dy_std=1.0, bn_params=True):
    """Inputs for an arbitrary layer spec (edge cases, ragged shapes): same recipe as 'bn'."""
    g = torch.Generator().manual_seed(seed)
    if x_dist == "uniform":
        x = torch.rand(spec.N, spec.H, spec.W, spec.IC, generator=g)
    else:
        x = torch.randn(spec.N, spec.H, spec.W, spec.IC, generator=g)
    fan = max(spec.fan_in, 1)
    li = _layer_params(g, spec, math.sqrt(2 / fan), 1 / math.sqrt(fan), bn_params)
    dy = torch.randn(spec.N, spec.OH, spec.OW, spec.OC, generator=g) * dy_std
    return dict(x=_round(x, spec.dtype), dy=_round(dy, spec.dtype), layers=[li])
