"""A training step captured in a CUDA graph replays to the same results as the eager calls.

The library's host work per call (tensor-map encoding, launch attributes) happens at capture time; the
graph holds the kernels with their programmatic dependencies. Both layers start from the same state, and
the kernels are deterministic, so every output must match bit for bit."""
import pytest
import torch

from conv2d_layer_gb300.abi import ACT_RELU, ACT_TANH, BF16, FP32, NORM_BATCH, NORM_NONE
from conv2d_layer_gb300.layer import Conv2dLayer
from conv2d_layer_gb300.workloads import LayerSpec, random_layer_inputs

CASES = {
    "bf16_bn_relu_pairs": LayerSpec(N=2, H=16, W=16, IC=64, OC=128, KH=3, KW=3, stride=1, pad=1, norm=NORM_BATCH,
                                    act=ACT_RELU, dtype=BF16),
    "fp32_tanh_s2": LayerSpec(N=2, H=15, W=13, IC=8, OC=24, KH=3, KW=3, stride=2, pad=1, norm=NORM_NONE,
                              act=ACT_TANH, dtype=FP32),
}


def _layer(spec, li):
    return Conv2dLayer(spec, li.w, li.b, li.gamma, li.beta, li.running_mean, li.running_var)


@pytest.mark.gpu
@pytest.mark.parametrize("name", list(CASES))
def test_training_step_replays_from_a_cuda_graph(name):
    spec = CASES[name]
    inp = random_layer_inputs(spec, 11)
    li = inp["layers"][0]
    x, dy = inp["x"].cuda(), inp["dy"].cuda()
    eager, graphed = _layer(spec, li), _layer(spec, li)

    eager.zero_grad()
    eager.fwd_train(x)
    eager.bwd(x, dy)

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        graphed.zero_grad()
        graphed.fwd_train(x)
        graphed.bwd(x, dy)
    g.replay()
    torch.cuda.synchronize()

    for k in ("y", "pre_act", "dx", "dw", "db", "dgamma", "dbeta", "running_mean", "running_var",
              "save_mean", "save_inv_std"):
        a, b = getattr(eager, k), getattr(graphed, k)
        assert torch.equal(a, b), k

    # a second replay is a second step: the running statistics move again, the gradients are recomputed
    # from zero (the graph holds the zeroing)
    rm1 = graphed.running_mean.clone()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(graphed.dw, eager.dw)
    if spec.norm == NORM_BATCH:
        assert not torch.equal(graphed.running_mean, rm1)
