"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every entry point include/conv2d.h declares, and rejects bad
arguments on the host (no kernel is launched when validation fails)."""
import ctypes
import os
import re

import pytest

from conv2d_layer_gb300 import abi

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "conv2d.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(conv2d_[a-z_0-9]+)\s*\(", src)))


def test_header_declares_the_binding_exports():
    assert _declared() == sorted(abi.EXPORTS)


def test_library_loads_and_exports_every_declared_symbol():
    L = abi.lib()
    for name in _declared():
        assert hasattr(L, name), name
        assert ctypes.cast(getattr(L, name), ctypes.c_void_p).value


def good(**kw):
    base = dict(N=2, H=8, W=8, IC=3, OC=4, KH=3, KW=3, stride=1, pad=1, norm=abi.NORM_BATCH, act=abi.ACT_RELU,
                dtype=abi.FP32, eps=1e-5, momentum=0.1)
    base.update(kw)
    return abi.desc(**base)


def test_out_hw():
    rc, oh, ow = abi.conv2d_out_hw(good(H=84, W=84, KH=8, KW=8, stride=4, pad=0))
    assert (rc, oh, ow) == (abi.OK, 20, 20)
    rc, oh, ow = abi.conv2d_out_hw(good(H=56, W=56, stride=2, pad=1))
    assert (rc, oh, ow) == (abi.OK, 28, 28)


@pytest.mark.parametrize("field,value,code", [
    ("N", 0, abi.ERR_INVALID_ARG), ("H", -1, abi.ERR_INVALID_ARG), ("IC", 0, abi.ERR_INVALID_ARG),
    ("OC", 0, abi.ERR_INVALID_ARG), ("KH", 0, abi.ERR_INVALID_ARG), ("stride", 0, abi.ERR_INVALID_ARG),
    ("pad", -1, abi.ERR_INVALID_ARG), ("KH", 11, abi.ERR_INVALID_ARG), ("norm", 4, abi.ERR_INVALID_ARG),
    ("act", 4, abi.ERR_INVALID_ARG), ("dtype", 2, abi.ERR_INVALID_ARG), ("eps", 0.0, abi.ERR_INVALID_ARG),
    ("eps", float("nan"), abi.ERR_INVALID_ARG), ("momentum", 1.5, abi.ERR_INVALID_ARG),
    ("momentum", -0.1, abi.ERR_INVALID_ARG), ("stride", 9, abi.ERR_UNSUPPORTED),
])
def test_validation_codes(field, value, code):
    d = good()
    setattr(d, field, value)
    assert abi.conv2d_validate(d) == code
    assert abi.conv2d_workspace_size(d, abi.OP_FWD_TRAIN) == 0


def test_eps_and_momentum_ignored_without_norm():
    assert abi.conv2d_validate(good(norm=abi.NORM_NONE, eps=0.0, momentum=7.0)) == abi.OK


def test_group_norm_groups_validated():
    assert abi.conv2d_validate(good(norm=abi.NORM_GROUP, groups=2)) == abi.OK       # OC = 4
    assert abi.conv2d_validate(good(norm=abi.NORM_GROUP, groups=3)) == abi.ERR_INVALID_ARG
    assert abi.conv2d_validate(good(norm=abi.NORM_GROUP, groups=0)) == abi.ERR_INVALID_ARG
    assert abi.conv2d_validate(good(norm=abi.NORM_LAYER, groups=0)) == abi.OK       # read for group norm only
    d = good(norm=abi.NORM_GROUP, groups=32, dtype=abi.BF16, H=56, W=56, IC=256, OC=256)
    for op in (abi.OP_FWD_TRAIN, abi.OP_FWD_INFER, abi.OP_BWD):
        assert abi.conv2d_workspace_size(d, op) > 0


def test_layer_norm_reads_eps_not_momentum():
    assert abi.conv2d_validate(good(norm=abi.NORM_LAYER)) == abi.OK
    assert abi.conv2d_validate(good(norm=abi.NORM_LAYER, momentum=7.0)) == abi.OK
    assert abi.conv2d_validate(good(norm=abi.NORM_LAYER, eps=0.0)) == abi.ERR_INVALID_ARG
    d = good(norm=abi.NORM_LAYER, dtype=abi.BF16, H=56, W=56, IC=256, OC=256)
    for op in (abi.OP_FWD_TRAIN, abi.OP_FWD_INFER, abi.OP_BWD):
        assert abi.conv2d_workspace_size(d, op) > 0


def test_workspace_sizes_positive_and_op_checked():
    d = good(dtype=abi.BF16, H=56, W=56, IC=256, OC=256)
    for op in (abi.OP_FWD_TRAIN, abi.OP_FWD_INFER, abi.OP_BWD):
        assert abi.conv2d_workspace_size(d, op) > 0
    assert abi.conv2d_workspace_size(d, 7) == 0
    # backward keeps d_conv (n_pix x OC operand elements) in the workspace
    assert abi.conv2d_workspace_size(d, abi.OP_BWD) >= 2 * 56 * 56 * 256 * 2


def test_fused_backward_keeps_no_dconv_tensor():
    # 1x1, stride-1 bf16 batch-norm layers with tanh or sigmoid form d_conv inside the dgrad and wgrad
    # producers: their backward workspace holds no n_pix x OC d_conv tensor; ReLU (and fp32, and a 3x3
    # kernel) keep it
    shape = dict(N=64, H=56, W=56, IC=128, OC=256, KH=1, KW=1, stride=1, pad=0, dtype=abi.BF16)
    dconv = 64 * 56 * 56 * 256 * 2
    fused = [abi.conv2d_workspace_size(good(act=a, **shape), abi.OP_BWD) for a in (abi.ACT_TANH, abi.ACT_SIGMOID)]
    kept = [abi.conv2d_workspace_size(good(**{**shape, **kw}), abi.OP_BWD)
            for kw in (dict(act=abi.ACT_RELU), dict(act=abi.ACT_TANH, dtype=abi.FP32),
                       dict(act=abi.ACT_TANH, KH=3, KW=3, pad=1), dict(act=abi.ACT_TANH, norm=abi.NORM_LAYER))]
    assert all(0 < f < dconv for f in fused)
    assert all(k >= dconv for k in kept)


def test_null_and_misaligned_pointers_rejected_before_launch():
    d = good(norm=abi.NORM_NONE)
    ws = ctypes.create_string_buffer(1 << 16)
    addr = ctypes.addressof(ws)
    al = (addr + 255) & ~255
    rc = abi.conv2d_fwd_train(d, None, al, None, None, None, None, None, al, None, None, al, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG
    rc = abi.conv2d_fwd_train(d, al + 4, al, None, None, None, None, None, al, None, None, al, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG
    dbn = good()
    rc = abi.conv2d_fwd_train(dbn, al, al, None, None, None, None, None, al, None, None, al, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG  # batch norm needs gamma, beta, running and saved statistics
    rc = abi.conv2d_bwd(d, al, al, None, None, al, None, None, al, None, None, None, None, None, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG  # neither dx nor dw requested
    dln = good(norm=abi.NORM_LAYER)
    rc = abi.conv2d_fwd_infer(dln, al, al, None, None, None, None, None, al, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG  # layer norm needs gamma, beta
    rc = abi.conv2d_fwd_train(dln, al, al, None, al, al, None, None, al, None, None, al, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG  # ... and the saved per-image statistics
    rc = abi.conv2d_bwd(dln, al, al, al, al, al, None, None, al, al, None, None, None, None, al, 1 << 15, 0)
    assert rc == abi.ERR_INVALID_ARG


def test_status_strings():
    for s in range(6):
        assert abi.status_str(s)
    assert abi.status_str(99) == "unknown status"


def test_layer_binding_rejects_mismatched_tensors_before_launch():
    """The C ABI trusts buffer sizes; Conv2dLayer checks every caller tensor first.

    A d_y drawn for a different layer (e.g. the last layer of a stack handed to
    the first) must raise, not reach a kernel that would read past its end."""
    import torch
    from conv2d_layer_gb300.layer import Conv2dLayer
    from conv2d_layer_gb300.workloads import LayerSpec
    spec = LayerSpec(N=2, H=8, W=8, IC=16, OC=32, KH=1, KW=1, stride=1, pad=0, norm=abi.NORM_BATCH,
                     act=abi.ACT_RELU, dtype=abi.BF16)
    L = Conv2dLayer(spec, torch.randn(32, 1, 1, 16), device="cpu")
    bf = torch.bfloat16
    good_x = torch.zeros(2, 8, 8, 16, dtype=bf)
    cases = [
        (lambda: L.fwd_train(torch.zeros(2, 8, 8, 8, dtype=bf)), "x: shape"),
        (lambda: L.fwd_train(good_x.float()), "x: dtype"),
        (lambda: L.fwd_train(torch.zeros(2, 16, 8, 8, dtype=bf).permute(0, 2, 3, 1)), "x: must be contiguous"),
        (lambda: L.fwd_train(good_x), "x: must be in CUDA device memory"),
        (lambda: L.fwd_train(None), "torch.Tensor"),
        (lambda: L.fwd_infer(good_x, y=torch.zeros(2, 8, 8, 16, dtype=bf)), "x: must be in CUDA"),
        (lambda: L.bwd(torch.zeros(1, 8, 8, 16, dtype=bf), torch.zeros(2, 8, 8, 32, dtype=bf)), "x: shape"),
    ]
    for call, msg in cases:
        with pytest.raises(ValueError, match=msg):
            call()


def test_layer_binding_tensor_check_rules():
    import torch
    from conv2d_layer_gb300.layer import _expect
    bf = torch.bfloat16
    # d_y of the last layer of the mixed stack (28x28) offered to its first layer (56x56)
    with pytest.raises(ValueError, match="dy: shape"):
        _expect(torch.zeros(2, 28, 28, 256, dtype=bf), "dy", (2, 56, 56, 256), bf)
    with pytest.raises(ValueError, match="y: shape"):
        _expect(torch.zeros(2, 8, 8, 15, dtype=bf), "y", (2, 8, 8, 16), bf)
    with pytest.raises(ValueError, match="CUDA"):
        _expect(torch.zeros(2, 3), "x", (2, 3), torch.float32)
    with pytest.raises(ValueError, match="torch.Tensor"):
        _expect(3, "x", (2, 3), torch.float32)
