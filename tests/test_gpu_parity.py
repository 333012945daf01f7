"""GPU parity: every step of the CUDA path, called through the C ABI, against
the CPU oracle on the same seeded inputs.

Bars: routing ids, offsets, sorted pairs, active list and count bit-exact;
routing weights within 1e-6; h and out within 1e-2 * max|oracle| + 1e-3
elementwise (the layer's stated tolerance)."""
import os

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


def run_layer(moe, logits, x, dw13, dw2, k):
    T, E = logits.shape
    layer = moe.MoELayer(dw13, dw2, T, k)
    lg = torch.from_numpy(logits).cuda()
    xx = torch.from_numpy(x).cuda()
    out = layer.forward(lg, xx)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(layer.workspace) == 0
    return layer, out


def check_meta(layer, ref, E):
    offs, sp, act, na = (t.cpu().numpy() for t in layer.meta)
    assert np.array_equal(offs, ref["expert_offsets"])
    assert np.array_equal(sp, ref["sorted_pair"])
    assert int(na[0]) == ref["num_active"]
    assert np.array_equal(act, ref["active_experts"])


# ------------------------------------------------------------------ routing
@pytest.mark.parametrize("T,E,k,hot", [(4, 16, 2, False), (8, 512, 10, False), (8, 512, 10, True),
                                       (4096, 512, 10, False), (33, 1024, 32, False),
                                       (5, 7, 7, False)])
def test_route_matches_oracle(moe, T, E, k, hot):
    logits = inputs.make_activations(T, 32, E, seed=T + E, hot_experts=range(16) if hot else (),
                                     hot_bias=2.0)[0]
    logits[0, :] = 0.0
    logits[0, 5] = -0.0             # -0 ties with +0: lower index first
    if T > 1:
        logits[1, 3] = logits[1, min(7, E - 1)] = 9.0   # planted tie at the top
    ids, w = moe.moe_topk_route(torch.from_numpy(logits).cuda(), k)
    ref_ids, ref_w = oracle.route(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=0, atol=1e-6)


# ------------------------------------------------------------------ grouping
@pytest.mark.parametrize("T,E,k", [(1, 512, 10), (8, 512, 10), (4, 16, 2), (127, 64, 6),
                                   (4096, 512, 10), (300, 1024, 32), (3, 4, 4)])
def test_align_matches_oracle(moe, T, E, k):
    ids = inputs.random_topk_ids(T, E, k, seed=T * 7 + k)
    meta = moe.moe_align_offsets(torch.from_numpy(ids).cuda(), E)
    offs, sp, act, na = (t.cpu().numpy() for t in meta)
    r_offs, r_sp, r_act, r_na = oracle.align(ids, E)
    assert np.array_equal(offs, r_offs)
    assert np.array_equal(sp, r_sp)
    assert int(na[0]) == r_na
    assert np.array_equal(act, r_act)


def test_align_empty_batch(moe):
    meta = moe.moe_align_offsets(torch.empty((0, 4), dtype=torch.int32, device="cuda"), 16)
    offs, sp, act, na = (t.cpu().numpy() for t in meta)
    assert np.all(offs == 0) and int(na[0]) == 0 and np.all(act == -1)


def test_align_flags_and_skips_bad_expert_id(moe):
    T, E, k = 6, 32, 4
    ids = inputs.random_topk_ids(T, E, k, seed=1)
    ids[2, 1] = E          # out of range: planted on the host
    ids[4, 0] = -3
    ws = moe.new_workspace(T, E, k, 32, 32)
    meta = moe.moe_align_offsets(torch.from_numpy(ids).cuda(), E, workspace=ws)
    flag = moe.moe_get_device_error(ws)
    assert flag & moe.MOE_DEVERR_BAD_EXPERT_ID
    offs, sp, act, na = (t.cpu().numpy() for t in meta)
    flat = ids.ravel()
    good = np.nonzero((flat >= 0) & (flat < E))[0]
    order = good[np.argsort(flat[good], kind="stable")]
    assert offs[E] == len(good)
    assert np.array_equal(sp[:len(good)], order)
    assert np.all(sp[len(good):] == -1)
    assert moe.moe_get_device_error(ws) == 0        # reading clears it


# ------------------------------------------------------------------ whole layer
LAYER_CASES = [
    inputs.TINY, inputs.QWEN_C1, inputs.QWEN_C2, inputs.QWEN_C4, inputs.QWEN_C8,
    inputs.TP4_C2, inputs.TP4_C4, inputs.TP4_C8,
    inputs.Workload("ragged_T5_H96_I96_E8_k3", inputs.MoEShape(5, 96, 96, 8, 3)),
    inputs.Workload("ragged_T3_H160_I32_E5_k5", inputs.MoEShape(3, 160, 32, 5, 5)),
    inputs.Workload("mid_T9_H512_I128_E64_k6", inputs.MoEShape(9, 512, 128, 64, 6)),
    inputs.Workload("mid_T127_H512_I128_E64_k6", inputs.MoEShape(127, 512, 128, 64, 6)),
    inputs.Workload("mid_T128_H512_I128_E64_k6", inputs.MoEShape(128, 512, 128, 64, 6)),
    inputs.Workload("skew_T64_H256_I64_E8_k2", inputs.MoEShape(64, 256, 64, 8, 2),
                    hot_experts=(3,), hot_bias=6.0),
]


@pytest.mark.parametrize("wl", LAYER_CASES, ids=lambda w: w.name)
def test_layer_matches_oracle(moe, wl):
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed, wl.hot_experts, wl.hot_bias)
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, wl.seed)
    layer, out = run_layer(moe, logits, x, dw13, dw2, sh.k)
    ref = oracle.moe_forward(logits, x, w13, w2, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ref["topk_ids"])
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), ref["topk_w"], rtol=0, atol=1e-6)
    check_meta(layer, ref, sh.E)
    assert_close(layer.h.float().cpu().numpy(), ref["h"], f"{wl.name} h")
    assert_close(out.float().cpu().numpy(), ref["out"], f"{wl.name} out")


def _oracle_rows(tokens, logits, x, w13, w2, k):
    """out rows of the given tokens from the oracle's per-token evaluation,
    spread over the host cores (each call is independent and releases the
    interpreter lock)."""
    import concurrent.futures as cf
    n = max(1, min(32, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(n) as pool:
        rows = list(pool.map(lambda t: oracle.moe_token(int(t), logits, x, w13, w2, k), tokens))
    return np.stack(rows)


def _check_h_rows(layer, tokens, ids_ref, x, w13, k, E):
    """h rows of every pair of the given tokens against the oracle's gate/up
    on sub-batches of those tokens (h of a pair depends on its token and
    expert only; the sub-batches run on the host cores).  The GPU's h is in
    sorted-row order of the full batch."""
    import concurrent.futures as cf
    tokens = np.asarray(tokens)
    sp_full = layer.meta[1].cpu().numpy()
    row_of_pair = np.empty_like(sp_full)
    row_of_pair[sp_full] = np.arange(len(sp_full), dtype=sp_full.dtype)
    h_gpu = layer.h.float().cpu().numpy()

    def part(toks):
        sub_meta = oracle.align(np.ascontiguousarray(ids_ref[toks]), E)
        rh = oracle.gate_up_silu(np.ascontiguousarray(x[toks]), w13, sub_meta, k)
        full_pairs = np.array([toks[p // k] * k + p % k for p in sub_meta[1]])
        return h_gpu[row_of_pair[full_pairs]], rh

    n = max(1, min(32, os.cpu_count() or 1))
    parts = np.array_split(tokens, max(1, min(len(tokens), 4 * n)))
    with cf.ThreadPoolExecutor(n) as pool:
        res = list(pool.map(part, [p for p in parts if len(p)]))
    assert_close(np.concatenate([g for g, _ in res]), np.concatenate([r for _, r in res]),
                 "h rows of the sampled tokens")


def _tokens_covering_every_chunk(sp, offs, act, na, k, per_chunk=2, chunk=128, min_rows=1):
    """Tokens whose pairs sit at the start and end of every 128-row chunk of
    every expert's segment of at least min_rows rows (so every tensor-core
    work item of those experts is checked)."""
    toks = set()
    for e in act[:na]:
        lo, hi = int(offs[e]), int(offs[e + 1])
        if hi - lo < min_rows:
            continue
        for c0 in range(lo, hi, chunk):
            c1 = min(hi, c0 + chunk)
            for r in list(range(c0, min(c1, c0 + per_chunk))) + list(range(max(c0, c1 - per_chunk), c1)):
                toks.add(int(sp[r]) // k)
    return sorted(toks)


def test_prefill_4096_every_token(moe):
    """The 4096-token workload at full size: routing and grouping bit-exact,
    every token's output against the oracle's per-token evaluation, and the
    h rows of the tokens at both ends of every tensor-core chunk."""
    wl = inputs.PREFILL
    sh = wl.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed)
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, wl.seed)
    layer, out = run_layer(moe, logits, x, dw13, dw2, sh.k)
    assert moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I) == moe.MOE_PATH_TENSOR_CORE
    ids_ref, w_ref = oracle.route(logits, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(layer.topk_w.cpu().numpy(), w_ref, rtol=0, atol=1e-6)
    r_offs, r_sp, r_act, r_na = oracle.align(ids_ref, sh.E)
    offs, sp, act, na = (t.cpu().numpy() for t in layer.meta)
    assert np.array_equal(offs, r_offs) and np.array_equal(sp, r_sp)
    assert np.array_equal(act, r_act) and int(na[0]) == r_na
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    ref = _oracle_rows(range(sh.T), logits, x, w13, w2, sh.k)
    assert_close(got, ref, "prefill out, every token")
    toks = _tokens_covering_every_chunk(r_sp, r_offs, r_act, r_na, sh.k, per_chunk=1)
    _check_h_rows(layer, toks, ids_ref, x, w13, sh.k, sh.E)


# Routing skewed so that hot experts' segments span several 128-row chunks of
# the tensor-core path (chunk index >= 1): all tokens checked at the small
# shape, and at the Qwen4Exp TP4-shard shape the tokens at both ends of every
# chunk plus their h rows.
def test_tensor_core_multi_chunk_segments_small(moe):
    wl = inputs.Workload("tcskew_T512_H512_I128_E16_k4_hot2", inputs.MoEShape(512, 512, 128, 16, 4),
                         hot_experts=(3, 9), hot_bias=6.0)
    sh = wl.shape
    assert moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I) == moe.MOE_PATH_TENSOR_CORE
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed, wl.hot_experts, wl.hot_bias)
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, wl.seed)
    layer, out = run_layer(moe, logits, x, dw13, dw2, sh.k)
    ref = oracle.moe_forward(logits, x, w13, w2, sh.k)
    offs = ref["expert_offsets"]
    assert max(np.diff(offs)) > 3 * 128          # a segment of four chunks
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ref["topk_ids"])
    check_meta(layer, ref, sh.E)
    assert_close(layer.h.float().cpu().numpy(), ref["h"], f"{wl.name} h")
    assert_close(out.float().cpu().numpy(), ref["out"], f"{wl.name} out")


def test_tensor_core_multi_chunk_segments_tp4_shape(moe):
    wl = inputs.Workload("tp4shard_T2048_H2560_I160_E512_k10_hot16", inputs.MoEShape(2048, 2560, 160, 512, 10),
                         hot_experts=tuple(range(16)), hot_bias=2.0)
    sh = wl.shape
    assert moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I) == moe.MOE_PATH_TENSOR_CORE
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, wl.seed, wl.hot_experts, wl.hot_bias)
    w13, w2, dw13, dw2 = weights(sh.E, sh.H, sh.I, wl.seed)
    layer, out = run_layer(moe, logits, x, dw13, dw2, sh.k)
    ids_ref, _ = oracle.route(logits, sh.k)
    assert np.array_equal(layer.topk_ids.cpu().numpy(), ids_ref)
    r_offs, r_sp, r_act, r_na = oracle.align(ids_ref, sh.E)
    offs, sp, act, na = (t.cpu().numpy() for t in layer.meta)
    assert np.array_equal(offs, r_offs) and np.array_equal(sp, r_sp)
    assert np.array_equal(act, r_act) and int(na[0]) == r_na
    assert max(np.diff(r_offs)) > 4 * 128        # hot segments of five or more chunks
    toks = _tokens_covering_every_chunk(r_sp, r_offs, r_act, r_na, sh.k, per_chunk=1)
    got = out.float().cpu().numpy()
    assert np.all(np.isfinite(got))
    assert_close(got[toks], _oracle_rows(toks, logits, x, w13, w2, sh.k), "tp4 T2048 out")
    # h: every chunk of the segments longer than one chunk
    long_toks = _tokens_covering_every_chunk(r_sp, r_offs, r_act, r_na, sh.k, per_chunk=2, min_rows=129)
    _check_h_rows(layer, long_toks, ids_ref, x, w13, sh.k, sh.E)


def test_decode_and_grouped_paths_agree_at_8_9_boundary(moe):
    """T = 8 (fused-combine decode kernels) and T = 9 (general path): the
    first eight tokens give the same outputs within tolerance."""
    sh = inputs.QWEN_C8.shape
    logits, x = inputs.make_activations(9, sh.H, sh.E, seed=11)
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    _, out9 = run_layer(moe, logits, x, dw13, dw2, sh.k)
    _, out8 = run_layer(moe, logits[:8], x[:8], dw13, dw2, sh.k)
    assert_close(out8.float().cpu().numpy(), out9[:8].float().cpu().numpy(), "T8 vs T9")


def test_zero_activation_gives_zero_output(moe):
    sh = inputs.QWEN_C4.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=2)
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    _, out = run_layer(moe, logits, np.zeros_like(x), dw13, dw2, sh.k)
    assert torch.count_nonzero(out).item() == 0


def test_repeated_calls_are_deterministic(moe):
    sh = inputs.QWEN_C8.shape
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=3)
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    a = layer.forward(lg, xx).clone()
    for _ in range(3):
        b = layer.forward(lg, xx)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert moe.moe_get_device_error(layer.workspace) == 0


def test_cuda_graph_capture_replay(moe):
    sh = inputs.QWEN_C2.shape
    _, _, dw13, dw2 = weights(sh.E, sh.H, sh.I, 0)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    lg = torch.zeros((sh.T, sh.E), dtype=torch.float32, device="cuda")
    xx = torch.zeros((sh.T, sh.H), dtype=torch.float16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer.forward(lg, xx)          # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer.forward(lg, xx)
    for seed in (4, 5):
        logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=seed)
        lg.copy_(torch.from_numpy(logits))
        xx.copy_(torch.from_numpy(x))
        g.replay()
        torch.cuda.synchronize()
        replayed = layer.out.clone()
        eager = layer.forward(lg, xx)
        torch.cuda.synchronize()
        assert torch.equal(replayed, eager)


def test_rejects_bad_arguments_without_launching(moe):
    x = torch.zeros((2, 64), dtype=torch.float32, device="cuda")
    with pytest.raises(moe.MoEError) as ei:
        moe.moe_topk_route(x, 65)            # k > E
    assert ei.value.status == moe.MOE_ERR_INVALID_ARG
    lib = moe.load_library()
    assert lib.moe_topk_route(x.data_ptr() + 4, 2, 64, 4, x.data_ptr(), x.data_ptr(),
                              None) == moe.MOE_ERR_INVALID_ARG   # misaligned


@pytest.mark.parametrize("T,E,k,hot", [(1, 512, 10, False), (8, 512, 10, False), (8, 512, 10, True),
                                       (32, 64, 6, False), (33, 64, 6, False), (4, 16, 2, False),
                                       (5, 7, 7, False), (2, 1024, 32, False)])
def test_route_align_fused_matches_oracle(moe, T, E, k, hot):
    """Steps 1-2 in one call (one launch for T <= 32, two kernels above)."""
    logits = inputs.make_activations(T, 32, E, seed=T * 3 + E, hot_experts=range(16) if hot else (),
                                     hot_bias=2.0)[0]
    if T > 1:
        logits[1, 2] = logits[1, min(5, E - 1)] = 7.5   # planted tie at the top
    ids, w, meta = moe.moe_topk_route_align(torch.from_numpy(logits).cuda(), k)
    ref_ids, ref_w = oracle.route(logits, k)
    assert np.array_equal(ids.cpu().numpy(), ref_ids)
    np.testing.assert_allclose(w.cpu().numpy(), ref_w, rtol=0, atol=1e-6)
    r_offs, r_sp, r_act, r_na = oracle.align(ref_ids, E)
    offs, sp, act, na = (t.cpu().numpy() for t in meta)
    assert np.array_equal(offs, r_offs) and np.array_equal(sp, r_sp)
    assert np.array_equal(act, r_act) and int(na[0]) == r_na


@pytest.mark.parametrize("T", [1, 3, 12])
def test_duplicate_experts_within_a_token(moe, T):
    """Caller-supplied ids may repeat an expert inside a token: segments then
    hold more rows than tokens.  Steps 2-4 against the oracle on the same ids
    and weights."""
    E, k, H, I = 16, 6, 256, 64
    rng = np.random.default_rng(T)
    ids = rng.integers(0, 4, size=(T, k)).astype(np.int32)      # heavy repeats
    ids[0, :] = 2                                               # one expert k times
    tw = rng.random((T, k)).astype(np.float32)
    x = inputs.make_activations(T, H, E, seed=T)[1]
    w13, w2, dw13, dw2 = weights(E, H, I, 0)
    ws = moe.new_workspace(T, E, k, H, I)
    meta = moe.moe_align_offsets(torch.from_numpy(ids).cuda(), E, workspace=ws)
    h = moe.moe_w4a16_gate_up_silu(torch.from_numpy(x).cuda(), dw13, meta, k, ws)
    out = moe.moe_w4a16_down_combine(h, dw2, meta, torch.from_numpy(tw).cuda(), ws)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) == 0
    rmeta = oracle.align(ids, E)
    for got, ref in zip(meta, rmeta[:3]):
        assert np.array_equal(got.cpu().numpy(), ref)
    rh = oracle.gate_up_silu(x, w13, rmeta, k)
    assert_close(h.float().cpu().numpy(), rh, "dup h")
    rout = oracle.down_combine(rh, w2, rmeta, tw.astype(np.float64), T, k)
    assert_close(out.float().cpu().numpy(), rout, "dup out")
