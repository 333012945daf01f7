"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself -- the binary16 format, hand-derived packed words, brute-force
dense evaluation, library routines (softmax, stable sort, matmul), closed
forms and invariants.  CPU only."""
import json
import math
import os

import numpy as np
import pytest
from scipy.special import softmax

from tests.dense_reference import moe_dense, route_dense, unpack_matrix
from w4a16_group_quantized_moe_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "dequant_words.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


# ---------------------------------------------------------------- binary16
def test_half_to_double_matches_numpy_for_every_bit_pattern(oracle_mod):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle_mod.half_to_double(int(b)) for b in bits])
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all((got == ref) | both_nan)
    assert np.array_equal(np.signbit(got[~both_nan]), np.signbit(ref[~both_nan]))


# ---------------------------------------------------------------- dequant
def _one_row_tensors(word, zword, scale=1.0, K=32, N=8):
    q = np.zeros((1, N, K // 8), np.uint32)
    q[0, :, 0] = word
    s = np.full((1, N, K // 32), scale, np.float16)
    z = np.zeros((1, N // 8, K // 32), np.uint32)
    z[0, 0, 0] = zword
    return q, s, z


def test_dequant_unpacks_hand_derived_words(oracle_mod):
    g = _golden()
    for case in g["qweight_words"]:
        q, s, z = _one_row_tensors(int(case["word"], 16), 0)
        for kk in range(8):
            assert oracle_mod.dequant(q, s, z, 8, 32, 0, 0, kk) == case["codes"][kk]
    for case in g["qzeros_words"]:
        q, s, z = _one_row_tensors(0, int(case["word"], 16))
        for n in range(8):
            assert oracle_mod.dequant(q, s, z, 8, 32, 0, n, 0) == -case["zeros_by_row_mod8"][n]


def test_dequant_applies_group_scale_and_zero(oracle_mod):
    # (q - z) * s with s = 0.0078125 (exact in fp16): q = 9 at kk = 1, z = 4 in row 0
    q, s, z = _one_row_tensors(0x00000090, 0x00000004, scale=0.0078125)
    assert oracle_mod.dequant(q, s, z, 8, 32, 0, 0, 1) == (9 - 4) * 0.0078125
    assert oracle_mod.dequant(q, s, z, 8, 32, 0, 0, 0) == (0 - 4) * 0.0078125
    assert oracle_mod.dequant(q, s, z, 8, 32, 0, 1, 1) == (9 - 0) * 0.0078125


def test_dequant_matches_dense_unpack_on_random_tensors(oracle_mod):
    w13, _ = inputs.make_weights(E=3, H=96, I=32, seed=5)
    dense = unpack_matrix(*w13)                         # [E][2I][H]
    rng = np.random.default_rng(0)
    for _ in range(400):
        e, n, kk = rng.integers(3), rng.integers(64), rng.integers(96)
        assert oracle_mod.dequant(*w13, 64, 96, int(e), int(n), int(kk)) == dense[e, n, kk]


# ---------------------------------------------------------------- routing
def test_route_hand_derived_cases(oracle_mod):
    for case in _golden()["route_cases"]:
        lg = np.array([case["logits"]], np.float32)
        ids, w = oracle_mod.route(lg, case["k"])
        assert ids[0].tolist() == case["ids"], case["why"]
        if "weights" in case:
            np.testing.assert_allclose(w[0], case["weights"], rtol=0, atol=1e-15)
    e6 = math.exp(6.0)
    ids, w = oracle_mod.route(np.array([[-1, 5, -1, -1, -1, -1, 5, -1]], np.float32), 3)
    np.testing.assert_allclose(w[0], np.array([e6, e6, 1.0]) / (2 * e6 + 1), rtol=1e-14)


@pytest.mark.parametrize("T,E,k", [(4, 16, 2), (7, 512, 10), (3, 33, 5), (2, 8, 8)])
def test_route_matches_brute_force_sort(oracle_mod, T, E, k):
    logits = np.random.default_rng(E + k).standard_normal((T, E)).astype(np.float32)
    logits[0, 3] = logits[0, 7] = logits[0].max() + 1.0      # planted tie at the top
    ids, w = oracle_mod.route(logits, k)
    ref_ids, ref_w = route_dense(logits, k)
    assert np.array_equal(ids, ref_ids)
    np.testing.assert_allclose(w, ref_w, rtol=1e-13, atol=0)
    assert ids[0, 0] == 3 and ids[0, 1] == 7


def test_route_k_equals_E_is_plain_softmax(oracle_mod):
    logits = np.random.default_rng(1).standard_normal((5, 24)).astype(np.float32)
    ids, w = oracle_mod.route(logits, 24)
    for t in range(5):
        np.testing.assert_allclose(w[t], softmax(logits[t].astype(np.float64))[ids[t]],
                                   rtol=1e-13)


def test_route_weights_positive_and_sum_to_one(oracle_mod):
    logits = inputs.make_activations(64, 32, 512, seed=3, hot_experts=range(16), hot_bias=2.0)[0]
    ids, w = oracle_mod.route(logits, 10)
    assert np.all(w > 0)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert all(len(set(r)) == 10 for r in ids.tolist())
    assert np.all(np.diff(np.take_along_axis(logits, ids, 1), axis=1) <= 0)


# ---------------------------------------------------------------- grouping
@pytest.mark.parametrize("T,E,k", [(4, 16, 2), (8, 512, 10), (300, 64, 6), (1, 4, 4)])
def test_align_matches_bincount_cumsum_and_stable_sort(oracle_mod, T, E, k):
    ids = inputs.random_topk_ids(T, E, k, seed=T)
    offs, sp, act, na = oracle_mod.align(ids, E)
    counts = np.bincount(ids.ravel(), minlength=E)
    assert np.array_equal(offs, np.concatenate([[0], np.cumsum(counts)]))
    assert np.array_equal(sp, np.argsort(ids.ravel(), kind="stable"))
    assert na == np.count_nonzero(counts)
    assert np.array_equal(act[:na], np.nonzero(counts)[0])
    assert np.all(act[na:] == -1)
    # partition invariant: every segment holds exactly its expert's pairs
    flat = ids.ravel()
    for e in range(E):
        seg = sp[offs[e]:offs[e + 1]]
        assert set(seg.tolist()) == set(np.nonzero(flat == e)[0].tolist())


def test_align_all_pairs_on_one_expert(oracle_mod):
    ids = np.zeros((5, 1), np.int32) + 3
    offs, sp, act, na = oracle_mod.align(ids, 6)
    assert offs.tolist() == [0, 0, 0, 0, 5, 5, 5]
    assert sp.tolist() == [0, 1, 2, 3, 4]
    assert na == 1 and act[0] == 3


# ---------------------------------------------------------------- full layer
SHAPES = [inputs.MoEShape(4, 256, 64, 16, 2),     # the tiny workload
          inputs.MoEShape(5, 96, 64, 8, 3),       # ragged: 3 groups along H
          inputs.MoEShape(3, 64, 32, 5, 5)]       # k = E, one group along I


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: f"T{s.T}H{s.H}I{s.I}E{s.E}k{s.k}")
def test_layer_matches_dense_brute_force(oracle_mod, sh):
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("t", sh))
    r = oracle_mod.moe_forward(logits, x, w13, w2, sh.k)
    out, h_dense, gate, ids, w = moe_dense(logits, x, w13, w2, sh.k)
    assert np.array_equal(r["topk_ids"], ids)
    np.testing.assert_allclose(r["topk_w"], w, rtol=1e-13)
    scale = np.abs(out).max()
    np.testing.assert_allclose(r["out"], out, rtol=0, atol=1e-11 * scale)
    # h rows in sorted order match the dense per-(expert, token) values
    for row, p in enumerate(r["sorted_pair"]):
        t, j = divmod(int(p), sh.k)
        e = r["topk_ids"][t, j]
        np.testing.assert_allclose(r["h"][row], h_dense[e, t], rtol=0,
                                   atol=1e-11 * np.abs(h_dense).max())


def test_layer_per_token_equals_batched(oracle_mod):
    sh = SHAPES[0]
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("t", sh))
    r = oracle_mod.moe_forward(logits, x, w13, w2, sh.k)
    for t in range(sh.T):
        assert np.array_equal(oracle_mod.moe_token(t, logits, x, w13, w2, sh.k), r["out"][t])
        one = oracle_mod.moe_forward(logits[t:t + 1], x[t:t + 1], w13, w2, sh.k)
        assert np.array_equal(one["out"][0], r["out"][t])       # batch invariance


def test_layer_zero_activation_gives_zero(oracle_mod):
    sh = SHAPES[0]
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("t", sh))
    r = oracle_mod.moe_forward(logits, np.zeros_like(x), w13, w2, sh.k)
    assert np.all(r["out"] == 0.0) and np.all(r["h"] == 0.0)


def _fill_codes(E, N, K, code):
    word = 0
    for j in range(8):
        word |= (code & 0xF) << (4 * j)
    return np.full((E, N, K // 8), word, np.uint32), np.full((E, N // 8, K // 32), word, np.uint32)


def test_layer_codes_equal_zeros_gives_zero(oracle_mod):
    sh = SHAPES[1]
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("t", sh))
    q13, z13 = _fill_codes(sh.E, 2 * sh.I, sh.H, 6)
    r = oracle_mod.moe_forward(logits, x, (q13, w13[1], z13), w2, sh.k)
    assert np.all(r["out"] == 0.0)


def test_layer_constant_closed_form(oracle_mod):
    # s = c, q - z = d, x = a everywhere: g = u = H*a*d*c, h = silu(g)*g,
    # y = I*h*d*c for every expert, and the renormalised weights sum to one.
    T, H, I, E, k = 3, 256, 64, 6, 3
    a, c, q, z = 0.5, 2.0 ** -7, 5, 2
    d = q - z
    qw13, _ = _fill_codes(E, 2 * I, H, q)
    _, zw13 = _fill_codes(E, 2 * I, H, z)
    qw2, _ = _fill_codes(E, H, I, q)
    _, zw2 = _fill_codes(E, H, I, z)
    w13 = (qw13, np.full((E, 2 * I, H // 32), c, np.float16), zw13)
    w2 = (qw2, np.full((E, H, I // 32), c, np.float16), zw2)
    logits = np.random.default_rng(2).standard_normal((T, E)).astype(np.float32)
    x = np.full((T, H), a, np.float16)
    r = oracle_mod.moe_forward(logits, x, w13, w2, k)
    g = H * a * d * c
    h = g / (1.0 + math.exp(-g)) * g
    y = I * h * d * c
    np.testing.assert_allclose(r["h"], h, rtol=1e-15)
    np.testing.assert_allclose(r["out"], y, rtol=1e-14)


def test_layer_single_expert_top1_is_dense_ffn(oracle_mod):
    T, H, I = 6, 128, 64
    logits = np.zeros((T, 1), np.float32)
    x = inputs.make_activations(T, H, 1, seed=9)[1]
    w13, w2 = inputs.make_weights(1, H, I, seed=9)
    W13 = unpack_matrix(*w13)[0]
    W2 = unpack_matrix(*w2)[0]
    xf = x.astype(np.float64)
    gu = xf @ W13.T
    ffn = (gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:]) @ W2.T
    r = oracle_mod.moe_forward(logits, x, w13, w2, 1)
    np.testing.assert_allclose(r["topk_w"], 1.0)
    np.testing.assert_allclose(r["out"], ffn, rtol=0, atol=1e-11 * np.abs(ffn).max())


def test_layer_invariant_under_expert_relabelling(oracle_mod):
    sh = SHAPES[0]
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("t", sh))
    perm = np.random.default_rng(4).permutation(sh.E)
    r = oracle_mod.moe_forward(logits, x, w13, w2, sh.k)
    rp = oracle_mod.moe_forward(logits[:, perm], x, tuple(a[perm] for a in w13),
                                tuple(a[perm] for a in w2), sh.k)
    assert np.array_equal(r["out"], rp["out"])
    assert np.array_equal(perm[rp["topk_ids"]], r["topk_ids"])
