"""GPU parity of the one-call layer (moe_w4a16_moe_layer) against the CPU
oracle: the one-launch decode layer for T <= 8 and the four-launch sequence
for larger batches.

Bars as for the step calls: routing ids bit-exact, routing weights within
1e-6, out within 1e-2 * max|oracle| + 1e-3 elementwise."""
import numpy as np
import pytest

import oracle
from w4a16_group_quantized_moe_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

TOL_REL, TOL_ABS = 1e-2, 1e-3


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import w4a16_group_quantized_moe_gb300 as m
    from w4a16_group_quantized_moe_gb300 import build
    build.build()
    m.load_library()
    return m


_WCACHE = {}


def weights(E, H, I, seed=0):
    key = (E, H, I, seed)
    if key not in _WCACHE:
        _WCACHE.clear()
        w13, w2 = inputs.make_weights(E, H, I, seed)
        from w4a16_group_quantized_moe_gb300 import to_device_weights
        _WCACHE[key] = (w13, w2, to_device_weights(w13), to_device_weights(w2))
    return _WCACHE[key]


def assert_close(got, ref, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    bound = TOL_REL * np.abs(ref).max() + TOL_ABS
    err = np.abs(got - ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    assert err.max() <= bound, f"{what}: max err {err.max():.3e} > bound {bound:.3e}"


def layer_call(moe, layer, logits, x):
    lg = torch.from_numpy(logits).cuda()
    xx = torch.from_numpy(x).cuda()
    out = layer.forward_layer(lg, xx)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(layer.workspace) == 0
    return out.float().cpu().numpy()


DECODE_CASES = [
    inputs.TINY, inputs.QWEN_C1, inputs.QWEN_C2, inputs.QWEN_C4, inputs.QWEN_C8,
    inputs.TP4_C2, inputs.TP4_C4, inputs.TP4_C8,
    inputs.Workload("ragged_T5_H96_I96_E8_k3", inputs.MoEShape(5, 96, 96, 8, 3)),
    inputs.Workload("ragged_T3_H160_I32_E5_k5", inputs.MoEShape(3, 160, 32, 5, 5)),
    inputs.Workload("mid_T8_H512_I128_E64_k6", inputs.MoEShape(8, 512, 128, 64, 6)),
    inputs.Workload("wide_T2_H1280_I320_E32_k4", inputs.MoEShape(2, 1280, 320, 32, 4)),
    inputs.Workload("wide_T4_H1280_I96_E32_k4", inputs.MoEShape(4, 1280, 96, 32, 4)),
    inputs.Workload("k32_T8_H256_I64_E1024_k32", inputs.MoEShape(8, 256, 64, 1024, 32)),
    inputs.Workload("skew_T8_H256_I64_E8_k2", inputs.MoEShape(8, 256, 64, 8, 2),
                    hot_experts=(3,), hot_bias=6.0),
]
OTHER_CASES = [
    inputs.Workload("mid_T9_H512_I128_E64_k6", inputs.MoEShape(9, 512, 128, 64, 6)),
    inputs.Workload("mid_T33_H512_I128_E64_k6", inputs.MoEShape(33, 512, 128, 64, 6)),
    inputs.Workload("tc_T128_H512_I128_E64_k6", inputs.MoEShape(128, 512, 128, 64, 6)),
    inputs.Workload("tc_T96_H256_I160_E16_k4", inputs.MoEShape(96, 256, 160, 16, 4),
                    hot_experts=(2, 5), hot_bias=3.0),
    # tensor-core edge cases: K blocks cut short (K = 96 is 1.5 blocks of 64)
    # and tiles past the last row; H = 384 leaves the second tile of the
    # last down item wholly past H
    inputs.Workload("tc_T80_H96_I96_E8_k3", inputs.MoEShape(80, 96, 96, 8, 3)),
    inputs.Workload("tc_T64_H384_I64_E16_k2", inputs.MoEShape(64, 384, 64, 16, 2)),
    # mid-size dispatch on the full hidden size: the decode step kernels,
    # with h read from global memory (too many rows to cache), at 9 tokens
    # with 14 warps, at 12 with 12 warps and at 16 with 10 (x rows of the
    # batch fill shared memory); 17 tokens (102 pairs at k = 6) the tensor
    # cores with one chunk cut short
    inputs.Workload("dec_T9_H2560_I640_E32_k10", inputs.MoEShape(9, 2560, 640, 32, 10)),
    inputs.Workload("dec_T12_H2560_I640_E32_k10", inputs.MoEShape(12, 2560, 640, 32, 10)),
    inputs.Workload("dec_T16_H2560_I640_E32_k10", inputs.MoEShape(16, 2560, 640, 32, 10)),
    inputs.Workload("tc_T17_H512_I128_E64_k6", inputs.MoEShape(17, 512, 128, 64, 6)),
]


@pytest.mark.parametrize("wl", DECODE_CASES + OTHER_CASES, ids=lambda w: w.name)
def test_layer_call_matches_oracle(moe, wl):
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed, wl.hot_experts, wl.hot_bias)
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, wl.seed)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    out = layer_call(moe, layer, logits, x)
    ref = oracle.moe_forward(logits, x, w13, w2, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ref["topk_ids"])
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), ref["topk_w"], rtol=0, atol=1e-6)
    assert_close(out, ref["out"], f"{wl.name} out")


def test_layer_call_consecutive_calls_share_the_workspace(moe):
    """Calls on one workspace with changing active experts: every call
    matches the oracle and a repeated input gives bit-identical output (the
    in-workspace counters are back at zero after each call)."""
    sh = inputs.QWEN_C4.shape
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    sets = [inputs.make_activations(sh.T, sh.H, sh.E, seed=s) for s in (21, 22, 23)]
    outs = [layer_call(moe, layer, lg, xx) for lg, xx in sets + sets[:1]]
    assert np.array_equal(outs[0], outs[3])
    for (lg, xx), o in zip(sets, outs):
        assert_close(o, oracle.moe_forward(lg, xx, w13, w2, sh.k)["out"], "consecutive")


def test_layer_call_agrees_with_step_calls(moe):
    sh = inputs.QWEN_C8.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=31)
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    fused = layer_call(moe, layer, logits, x)
    ids = layer.topk_ids.clone()
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    steps = layer.forward(lg, xx).float().cpu().numpy()
    assert torch.equal(ids, layer.topk_ids)
    assert_close(fused, steps, "one call vs four calls")


def test_layer_call_zero_activation_gives_zero_output(moe):
    sh = inputs.QWEN_C2.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=2)
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    out = layer_call(moe, layer, logits, np.zeros_like(x))
    assert not np.any(out)


def test_layer_call_empty_batch_is_a_no_op(moe):
    sh = inputs.QWEN_C1.shape
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    ws = moe.new_layer_workspace(1, sh.E, sh.k, sh.H, sh.I)
    lg = torch.empty((0, sh.E), dtype=torch.float32, device="cuda")
    xx = torch.empty((0, sh.H), dtype=torch.float16, device="cuda")
    out, ids, w = moe.moe_w4a16_moe_layer(lg, xx, dw13, dw2, sh.k, ws)
    torch.cuda.synchronize()
    assert out.shape == (0, sh.H) and ids.shape == (0, sh.k)


def test_layer_call_rejects_small_workspace(moe):
    sh = inputs.QWEN_C1.shape
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=1)
    small = moe.new_workspace(sh.T, sh.E, sh.k, sh.H, sh.I)  # the step calls' size only
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_w4a16_moe_layer(torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda(),
                                dw13, dw2, sh.k, small)
    assert ei.value.status == moe.MOE_ERR_WORKSPACE
