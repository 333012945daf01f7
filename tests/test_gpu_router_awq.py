"""GPU parity for the steps on either side of the layer, through the C ABI:
router logits (GEMV and tensor-core paths) and the fused router + routing +
grouping call against the oracle, and the AWQ checkpoint import bit for bit.

Bars: logits within the worst-case bound of an fp32 sum of exact fp16
products, |err| <= H * 2^-24 * sum_h |x_h w_h| (+1e-30); routing of the GPU's
own logits bit-exact against the oracle's router applied to those logits
(weights within 1e-6), grouping bit-exact; the import bit-exact."""
import numpy as np
import pytest

import oracle
from tests.test_gpu_parity import assert_close, moe  # noqa: F401
from w4a16_group_quantized_moe_gb300 import inputs

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _logit_bound(x, wr):
    a = np.abs(x.astype(np.float64)) @ np.abs(wr.astype(np.float64)).T
    return x.shape[1] * 2.0 ** -24 * a + 1e-30


def _check_logits(got, x, wr, rows=None):
    rows = np.arange(x.shape[0]) if rows is None else np.asarray(rows)
    ref = oracle.router_logits(x[rows], wr)
    err = np.abs(got[rows].astype(np.float64) - ref)
    bound = _logit_bound(x[rows], wr)
    assert np.all(np.isfinite(got[rows]))
    assert np.all(err <= bound), f"logit err {err.max():.3e} above its bound at {np.unravel_index((err - bound).argmax(), err.shape)}"


# (T, E, H): GEMV band (T <= 16), tensor cores above; ragged E and H (H not a
# multiple of the 64-wide K block, E not a multiple of the 128-expert tile)
LOGIT_CASES = [(1, 512, 2560), (2, 512, 2560), (5, 512, 2560), (8, 512, 2560), (16, 512, 2560),
               (3, 100, 96), (16, 1024, 160), (17, 512, 2560), (128, 512, 2560), (300, 100, 96),
               (257, 130, 2560), (1000, 16, 256)]


@pytest.mark.parametrize("T,E,H", LOGIT_CASES, ids=lambda v: str(v))
def test_router_logits_match_oracle(moe, T, E, H):
    x = inputs.make_activations(T, H, E, seed=T)[1]
    wr = inputs.make_router(E, H, seed=T)
    got = moe.moe_router_logits(torch.from_numpy(x).cuda(), torch.from_numpy(wr).cuda())
    torch.cuda.synchronize()
    _check_logits(got.cpu().numpy(), x, wr)


def test_router_logits_prefill_sampled(moe):
    """The 4096-token batch on the tensor cores: every 128-token tile's
    first and last rows and a random sample against the oracle."""
    T, E, H = 4096, 512, 2560
    x = inputs.make_activations(T, H, E, seed=7)[1]
    wr = inputs.make_router(E, H, seed=7)
    got = moe.moe_router_logits(torch.from_numpy(x).cuda(), torch.from_numpy(wr).cuda())
    torch.cuda.synchronize()
    rows = sorted(set(list(range(0, T, 128)) + list(range(127, T, 128)) +
                      list(np.random.default_rng(0).choice(T, 64, replace=False))))
    _check_logits(got.cpu().numpy(), x, wr, rows)


@pytest.mark.parametrize("T,E,k,H", [(1, 512, 10, 2560), (4, 512, 10, 2560), (8, 512, 10, 2560),
                                     (16, 512, 10, 2560), (3, 16, 2, 256), (16, 1024, 32, 96),
                                     (17, 512, 10, 2560), (64, 512, 10, 2560), (4096, 512, 10, 2560)],
                         ids=lambda v: str(v))
def test_router_route_align_matches_oracle(moe, T, E, k, H):
    x = inputs.make_activations(T, H, E, seed=T + 1)[1]
    wr = inputs.make_router(E, H, seed=T + 1)
    ws = moe.new_workspace(T, E, k, H, 32)
    xd, wd = torch.from_numpy(x).cuda(), torch.from_numpy(wr).cuda()
    for call in range(2):  # the second call reuses the workspace (ticket left at zero)
        logits, ids, w, meta = moe.moe_router_route_align(xd, wd, k, ws)
        torch.cuda.synchronize()
        assert moe.moe_get_device_error(ws) == 0
    lg = logits.cpu().numpy()
    rows = np.arange(T) if T <= 64 else np.unique(np.r_[np.arange(0, T, 97), T - 1])
    _check_logits(lg, x, wr, rows)
    ids_ref, w_ref = oracle.route(lg, k)
    assert np.array_equal(ids.cpu().numpy(), ids_ref)
    np.testing.assert_allclose(w.cpu().numpy(), w_ref, rtol=0, atol=1e-6)
    r_offs, r_sp, r_act, r_na = oracle.align(ids_ref, E)
    offs, sp, act, na = (t.cpu().numpy() for t in meta)
    assert np.array_equal(offs, r_offs) and np.array_equal(sp, r_sp)
    assert np.array_equal(act, r_act) and int(na[0]) == r_na


def test_router_route_align_in_a_graph(moe):
    """The fused one-launch router captured in a CUDA graph and replayed
    three times on new inputs gives the eager results."""
    T, E, k, H = 8, 512, 10, 2560
    wd = torch.from_numpy(inputs.make_router(E, H)).cuda()
    xs = [torch.from_numpy(inputs.make_activations(T, H, E, seed=s)[1]).cuda() for s in range(3)]
    ws = moe.new_workspace(T, E, k, H, 32)
    eager = [tuple(t.clone() for t in moe.moe_router_route_align(xx, wd, k, ws)[:3]) for xx in xs]
    xin = xs[0].clone()
    lg, ids, w, meta = moe.moe_router_route_align(xin, wd, k, ws)
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        moe.moe_router_route_align(xin, wd, k, ws, logits=lg, topk_ids=ids, topk_w=w, meta=meta, stream=s)
    for xx, (e_lg, e_ids, e_w) in zip(xs, eager):
        xin.copy_(xx)
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(lg, e_lg) and torch.equal(ids, e_ids) and torch.equal(w, e_w)
    assert moe.moe_get_device_error(ws) == 0


# ---------------------------------------------------------------- AWQ import
def _dev_awq(awq):
    aq, az, as_ = awq
    return (torch.from_numpy(aq.view(np.int32)).cuda(), torch.from_numpy(az.view(np.int32)).cuda(),
            torch.from_numpy(as_).cuda())


def _sentinel_dst(E, Ndst, K, seed):
    rng = np.random.default_rng(seed)
    return (rng.integers(0, 1 << 32, (E, Ndst, K // 8), dtype=np.uint32),
            rng.random((E, Ndst, K // 32)).astype(np.float16),
            rng.integers(0, 1 << 32, (E, Ndst // 8, K // 32), dtype=np.uint32))


def _to_dev(dst):
    q, s, z = dst
    return (torch.from_numpy(q.view(np.int32).copy()).cuda(), torch.from_numpy(s.copy()).cuda(),
            torch.from_numpy(z.view(np.int32).copy()).cuda())


def _from_dev(dd):
    q, s, z = (t.cpu().numpy() for t in dd)
    return q.view(np.uint32), s, z.view(np.uint32)


# (E, K, N, Ndst, row0): gate/up halves of W13 and the down matrix at the
# Qwen4Exp shapes (few experts), the TP4 shard, and ragged tiles (K not a
# multiple of the 256-row tile, N not of the 64-column tile)
AWQ_CASES = [(4, 2560, 640, 1280, 0), (4, 2560, 640, 1280, 640), (4, 640, 2560, 2560, 0),
             (3, 2560, 160, 320, 160), (2, 96, 40, 48, 8), (5, 288, 72, 72, 0), (1, 32, 8, 16, 8)]


@pytest.mark.parametrize("E,K,N,Ndst,row0", AWQ_CASES, ids=lambda v: str(v))
def test_awq_import_bit_exact(moe, E, K, N, Ndst, row0):
    awq = inputs.make_awq_layer(E, K, N, seed=K + N)
    dst = _sentinel_dst(E, Ndst, K, seed=E + K)
    ref = oracle.awq_import(awq, tuple(a.copy() for a in dst), row0)
    dd = _to_dev(dst)
    moe.moe_awq_import(_dev_awq(awq), dd, row0)
    torch.cuda.synchronize()
    for g, r, name in zip(_from_dev(dd), ref, ("qweight", "scales", "qzeros")):
        assert np.array_equal(g.view(np.uint16) if name == "scales" else g,
                              r.view(np.uint16) if name == "scales" else r), name


def test_awq_import_full_expert_count_sampled(moe):
    """All 512 experts of a Qwen4Exp gate layer imported on the GPU; eight
    experts spread over the stack against the oracle's import of those."""
    E, K, N = 512, 2560, 640
    awq = inputs.make_awq_layer(E, K, N, seed=3)
    dd = tuple(torch.zeros(shape, dtype=dt, device="cuda") for shape, dt in
               (((E, 2 * N, K // 8), torch.int32), ((E, 2 * N, K // 32), torch.float16),
                ((E, 2 * N // 8, K // 32), torch.int32)))
    moe.moe_awq_import(_dev_awq(awq), dd, 0)
    torch.cuda.synchronize()
    for e in (0, 1, 77, 255, 256, 300, 510, 511):
        sub = tuple(a[e:e + 1] for a in awq)
        ref = oracle.awq_import(sub, (np.zeros((1, 2 * N, K // 8), np.uint32), np.zeros((1, 2 * N, K // 32), np.float16),
                                      np.zeros((1, 2 * N // 8, K // 32), np.uint32)), 0)
        got = tuple(t[e:e + 1].cpu().numpy() for t in dd)
        assert np.array_equal(got[0].view(np.uint32), ref[0])
        assert np.array_equal(got[1].view(np.uint16), ref[1].view(np.uint16))
        assert np.array_equal(got[2].view(np.uint32), ref[2])


def test_awq_checkpoint_to_layer_output(moe):
    """Gate, up and down AWQ layers imported on the GPU into W13 and W2, then
    the layer run on them: out against the oracle's layer on the oracle's
    import of the same checkpoint."""
    T, H, I, E, k = 4, 256, 64, 16, 2
    gate, up = inputs.make_awq_layer(E, H, I, seed=1, tag=61), inputs.make_awq_layer(E, H, I, seed=1, tag=71)
    down = inputs.make_awq_layer(E, I, H, seed=1, tag=81)
    w13 = oracle.awq_import(up, oracle.awq_import(gate, (np.zeros((E, 2 * I, H // 8), np.uint32),
                                                         np.zeros((E, 2 * I, H // 32), np.float16),
                                                         np.zeros((E, 2 * I // 8, H // 32), np.uint32)), 0), I)
    w2 = oracle.awq_import(down, (np.zeros((E, H, I // 8), np.uint32), np.zeros((E, H, I // 32), np.float16),
                                  np.zeros((E, H // 8, I // 32), np.uint32)), 0)
    d13 = tuple(torch.zeros(a.shape, dtype=torch.float16 if a.dtype == np.float16 else torch.int32, device="cuda")
                for a in w13)
    d2 = tuple(torch.zeros(a.shape, dtype=torch.float16 if a.dtype == np.float16 else torch.int32, device="cuda")
               for a in w2)
    moe.moe_awq_import(_dev_awq(gate), d13, 0)
    moe.moe_awq_import(_dev_awq(up), d13, I)
    moe.moe_awq_import(_dev_awq(down), d2, 0)
    logits, x = inputs.make_activations(T, H, E, 0)
    layer = moe.MoELayer(d13, d2, T, k)
    out = layer.forward(torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda())
    torch.cuda.synchronize()
    ref = oracle.moe_forward(logits, x, w13, w2, k)
    assert_close(out.float().cpu().numpy(), ref["out"], "layer on imported AWQ weights")


def test_awq_import_rejects_bad_placement(moe):
    awq = _dev_awq(inputs.make_awq_layer(1, 64, 16))
    dst = _to_dev(_sentinel_dst(1, 32, 64, 0))
    for row0 in (4, 24):  # not a multiple of 8; rows past the end
        with pytest.raises(moe.MoEError) as ei:
            moe.moe_awq_import(awq, dst, row0)
        assert ei.value.status == moe.MOE_ERR_INVALID_ARG
