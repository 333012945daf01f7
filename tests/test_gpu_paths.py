"""Every kernel family of the step calls, forced through the _ex calls, at
shapes on both sides of the dispatch boundaries, against the oracle; the two
steps on different families; forced paths a shape cannot take rejected
before any launch.  Bars as in test_gpu_parity."""
import numpy as np
import pytest

import oracle
from tests.test_gpu_parity import assert_close, check_meta, moe, weights  # noqa: F401
from w4a16_group_quantized_moe_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

W = inputs.Workload
PATH_CASES = [
    inputs.TINY,
    W("b_T8_H512_I128_E64_k6", inputs.MoEShape(8, 512, 128, 64, 6)),
    W("b_T9_H512_I128_E64_k6", inputs.MoEShape(9, 512, 128, 64, 6)),
    W("b_T16_H512_I128_E64_k6", inputs.MoEShape(16, 512, 128, 64, 6)),
    W("b_T17_H512_I128_E64_k6", inputs.MoEShape(17, 512, 128, 64, 6)),
    W("b_T40_H256_I64_E8_k2", inputs.MoEShape(40, 256, 64, 8, 2)),
    W("b_T127_H512_I128_E64_k6", inputs.MoEShape(127, 512, 128, 64, 6)),
    inputs.QWEN_C8,
    W("qwen4exp_T12_H2560_I640_E512_k10", inputs.MoEShape(12, 2560, 640, 512, 10)),
    W("qwen4exp_T16_H2560_I640_E512_k10", inputs.MoEShape(16, 2560, 640, 512, 10)),
    W("qwen4exp_T24_H2560_I640_E512_k10", inputs.MoEShape(24, 2560, 640, 512, 10)),
    inputs.TP4_C8,
]
PATHS = {"decode": 1, "tensor_core": 2, "stream": 3}


def _run(moe, wl, gu_path, dn_path):
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed, wl.hot_experts, wl.hot_bias)
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, wl.seed)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    moe.moe_topk_route(lg, sh.k, layer.topk_ids, layer.topk_w)
    moe.moe_align_offsets(layer.topk_ids, sh.E, layer.workspace, out=layer.meta)
    try:
        moe.moe_w4a16_gate_up_silu(xx, dw13, layer.meta, sh.k, layer.workspace, h=layer.h, path=gu_path)
        moe.moe_w4a16_down_combine(layer.h, dw2, layer.meta, layer.topk_w, layer.workspace, out=layer.out,
                                   path=dn_path)
    except moe.MoEError as e:
        if e.status == moe.MOE_ERR_UNSUPPORTED:
            pytest.skip("the forced family does not take this shape")
        raise
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(layer.workspace) == 0
    return logits, x, w13, w2, layer


@pytest.mark.parametrize("path", list(PATHS), ids=list(PATHS))
@pytest.mark.parametrize("wl", PATH_CASES, ids=lambda w: w.name)
def test_forced_path_matches_oracle(moe, wl, path):
    sh = wl.shape
    p = PATHS[path]
    logits, x, w13, w2, layer = _run(moe, wl, p, p)
    ref = oracle.moe_forward(logits, x, w13, w2, sh.k)
    check_meta(layer, ref, sh.E)
    assert_close(layer.h.float().cpu().numpy(), ref["h"], f"{wl.name} {path} h")
    assert_close(layer.out.float().cpu().numpy(), ref["out"], f"{wl.name} {path} out")


@pytest.mark.parametrize("gu,dn", [("decode", "stream"), ("stream", "decode"), ("tensor_core", "stream"),
                                   ("stream", "tensor_core"), ("decode", "tensor_core")])
def test_steps_on_different_paths(moe, gu, dn):
    wl = PATH_CASES[3]  # T = 16: every family takes it
    sh = wl.shape
    logits, x, w13, w2, layer = _run(moe, wl, PATHS[gu], PATHS[dn])
    ref = oracle.moe_forward(logits, x, w13, w2, sh.k)
    assert_close(layer.out.float().cpu().numpy(), ref["out"], f"{gu} then {dn}")


def test_forced_path_rejections(moe):
    """Decode kernels at 4096 tokens and the tensor cores at 4 tokens cannot
    take the shape: MOE_ERR_UNSUPPORTED, nothing written; an unknown path
    value is MOE_ERR_INVALID_ARG."""
    for T, path in ((4096, moe.MOE_PATH_DECODE), (4, moe.MOE_PATH_TENSOR_CORE)):
        E, k, H, I = 64, 6, 512, 128
        _, _, dw13, _ = weights(E, H, I, 0)
        layer = moe.MoELayer(dw13, dw13, T, k)
        layer.h.fill_(3.0)
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_w4a16_gate_up_silu(torch.zeros((T, H), dtype=torch.float16, device="cuda"), dw13, layer.meta,
                                       k, layer.workspace, h=layer.h, path=path)
        assert ei.value.status == moe.MOE_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        assert torch.all(layer.h == 3.0)
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_w4a16_gate_up_silu(torch.zeros((4, H), dtype=torch.float16, device="cuda"), dw13, layer.meta, k,
                                   moe.new_workspace(4, E, k, H, I), h=torch.empty((4 * k, I), dtype=torch.float16,
                                                                                   device="cuda"), path=7)
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG


def test_auto_path_is_the_reported_path(moe):
    """The path moe_step_kernel_path reports is the one AUTO runs: forcing it
    gives the AUTO result bit for bit."""
    for wl in (PATH_CASES[2], PATH_CASES[5], PATH_CASES[8], inputs.QWEN_C1):
        sh = wl.shape
        p = moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I)
        assert p in (1, 2, 3)
        _, _, _, _, a = _run(moe, wl, moe.MOE_PATH_AUTO, moe.MOE_PATH_AUTO)
        _, _, _, _, f = _run(moe, wl, p, p)
        assert torch.equal(a.h, f.h) and torch.equal(a.out, f.out)
