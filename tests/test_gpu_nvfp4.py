"""GPU parity for the NVFP4-weight calls (E2M1 codes, E4M3 scales per 16
elements along K, fp32 scale per expert matrix, fp16 activations), through
the C ABI, against the oracle's NVFP4 functions on the same seeded inputs.

Bars as for W4A16: routing and grouping bit-exact, h and out within
1e-2 * max|oracle| + 1e-3 elementwise."""
import numpy as np
import pytest

import oracle
from tests.test_gpu_parity import (LAYER_CASES, _tokens_covering_every_chunk, assert_close, moe)  # noqa: F401
from w4a16_group_quantized_moe_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

_WCACHE = {}


def weights_nvfp4(E, H, I, seed=0):
    key = (E, H, I, seed)
    if key not in _WCACHE:
        _WCACHE.clear()
        w13, w2 = inputs.make_weights_nvfp4(E, H, I, seed)
        from w4a16_group_quantized_moe_gb300 import to_device_weights_nvfp4
        _WCACHE[key] = (w13, w2, to_device_weights_nvfp4(w13), to_device_weights_nvfp4(w2))
    return _WCACHE[key]


def _layer(moe, wl, one_call):
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed, wl.hot_experts, wl.hot_bias)
    w13, w2, dw13, dw2 = weights_nvfp4(sh.E, sh.H, sh.I, wl.seed)
    layer = moe.MoELayerNvfp4(dw13, dw2, sh.T, sh.k)
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    out = layer.forward_layer(lg, xx) if one_call else layer.forward(lg, xx)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(layer.workspace) == 0
    return logits, x, w13, w2, layer, out


# every W4A16 layer case, plus segments of four 128-row chunks on the tensor cores
NV_CASES = LAYER_CASES + [
    inputs.Workload("tcskew_T512_H512_I128_E16_k4_hot2", inputs.MoEShape(512, 512, 128, 16, 4),
                    hot_experts=(3, 9), hot_bias=6.0),
]


@pytest.mark.parametrize("one_call", [False, True], ids=["steps", "one_call"])
@pytest.mark.parametrize("wl", NV_CASES, ids=lambda w: w.name)
def test_nvfp4_layer_matches_oracle(moe, wl, one_call):
    sh = wl.shape
    path = moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I)
    assert path in (moe.MOE_PATH_DECODE, moe.MOE_PATH_TENSOR_CORE)
    logits, x, w13, w2, layer, out = _layer(moe, wl, one_call)
    ref = oracle.moe_forward_nvfp4(logits, x, w13, w2, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ref["topk_ids"])
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), ref["topk_w"], rtol=0, atol=1e-6)
    if not one_call:  # the fused layer keeps its h rows in the workspace
        offs, sp, act, na = (t.cpu().numpy() for t in layer.meta)
        assert np.array_equal(offs, ref["expert_offsets"]) and np.array_equal(sp, ref["sorted_pair"])
        assert_close(layer.h.float().cpu().numpy(), ref["h"], f"{wl.name} h")
    assert_close(out.float().cpu().numpy(), ref["out"], f"{wl.name} out")


def _oracle_rows_nvfp4(tokens, logits, x, w13, w2, k):
    import concurrent.futures as cf
    import os
    n = max(1, min(32, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(n) as pool:
        rows = list(pool.map(lambda t: oracle.moe_token_nvfp4(int(t), logits, x, w13, w2, k), tokens))
    return np.stack(rows)


@pytest.mark.parametrize("wl", [
    inputs.PREFILL,
    inputs.Workload("tp4shard_T2048_H2560_I160_E512_k10_hot16", inputs.MoEShape(2048, 2560, 160, 512, 10),
                    hot_experts=tuple(range(16)), hot_bias=2.0),
], ids=lambda w: w.name)
def test_nvfp4_tensor_core_full_size_sampled(moe, wl):
    """Full-size tensor-core workloads: routing and grouping bit-exact, out
    of the tokens at both ends of every 128-row chunk of every segment
    against the oracle's per-token evaluation, and h of those tokens against
    the oracle's gate/up on a sub-batch."""
    sh = wl.shape
    assert moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I) == moe.MOE_PATH_TENSOR_CORE
    logits, x, w13, w2, layer, out = _layer(moe, wl, one_call=False)
    ids_ref, _ = oracle.route(logits, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    r_offs, r_sp, r_act, r_na = oracle.align(ids_ref, sh.E)
    offs, sp, act, na = (t.cpu().numpy() for t in layer.meta)
    assert np.array_equal(offs, r_offs) and np.array_equal(sp, r_sp)
    toks = _tokens_covering_every_chunk(r_sp, r_offs, r_act, r_na, sh.k, per_chunk=1)
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert_close(got[toks], _oracle_rows_nvfp4(toks, logits, x, w13, w2, sh.k), f"{wl.name} out")
    # h rows: the sampled tokens as one sub-batch, mapped to the full batch's sorted rows
    sub = np.asarray(toks[:256])
    sub_meta = oracle.align(np.ascontiguousarray(ids_ref[sub]), sh.E)
    rh = oracle.gate_up_silu_nvfp4(np.ascontiguousarray(x[sub]), w13, sub_meta, sh.k)
    row_of_pair = np.empty_like(sp)
    row_of_pair[sp] = np.arange(len(sp), dtype=sp.dtype)
    full_pairs = np.array([sub[p // sh.k] * sh.k + p % sh.k for p in sub_meta[1]])
    assert_close(layer.h.float().cpu().numpy()[row_of_pair[full_pairs]], rh, f"{wl.name} h rows")


@pytest.mark.parametrize("one_call", [False, True], ids=["steps", "one_call"])
def test_nvfp4_between_decode_and_full_chunks(moe, one_call):
    """T = 40, k = 2 (P = 80): past the decode kernels and short of one
    128-row chunk, so the tensor cores run with chunks cut short."""
    wl = inputs.Workload("mid_T40_H256_I64_E8_k2", inputs.MoEShape(40, 256, 64, 8, 2))
    sh = wl.shape
    assert moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I) == moe.MOE_PATH_TENSOR_CORE
    logits, x, w13, w2, layer, out = _layer(moe, wl, one_call)
    ref = oracle.moe_forward_nvfp4(logits, x, w13, w2, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ref["topk_ids"])
    assert_close(out.float().cpu().numpy(), ref["out"], f"{wl.name} out")


def test_nvfp4_zero_expert_scale_zeroes_the_expert(moe):
    """gscale = 0 for every gate/up matrix: h and out are exactly zero (a
    closed form that needs no oracle); with the down scales alone zeroed,
    out is exactly zero."""
    wl = inputs.QWEN_C4
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed)
    _, _, dw13, dw2 = weights_nvfp4(sh.E, sh.H, sh.I, wl.seed)
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    z13 = (dw13[0], dw13[1], torch.zeros_like(dw13[2]))
    layer = moe.MoELayerNvfp4(z13, dw2, sh.T, sh.k)
    out = layer.forward(lg, xx)
    torch.cuda.synchronize()
    assert torch.count_nonzero(layer.h) == 0 and torch.count_nonzero(out) == 0
    z2 = (dw2[0], dw2[1], torch.zeros_like(dw2[2]))
    layer = moe.MoELayerNvfp4(dw13, z2, sh.T, sh.k)
    out = layer.forward_layer(lg, xx)
    torch.cuda.synchronize()
    assert torch.count_nonzero(out) == 0


def test_nvfp4_graph_capture_replay(moe):
    """The one-call NVFP4 layer captured in a CUDA graph and replayed gives
    the eager result bit for bit."""
    wl = inputs.QWEN_C8
    sh = wl.shape
    logits, x, _, _, layer, out = _layer(moe, wl, one_call=True)
    eager = out.clone()
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    layer.out.zero_()
    with torch.cuda.graph(g, stream=s):
        layer.forward_layer(lg, xx, stream=s)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(layer.out, eager)
