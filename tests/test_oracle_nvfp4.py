"""Pins for the oracle's NVFP4 weight format (E2M1 codes, E4M3 scales per 16
elements along K, an fp32 scale per expert matrix; fp16 activations): the
E2M1 value table of the OCP Microscaling specification, PyTorch's own
float8_e4m3fn decoding of every byte, hand-derived words, a dense numpy
brute force with those independent decoders, a closed form and per-token
consistency.  CPU only."""
import numpy as np
import pytest

from tests.dense_reference import E2M1_VALUES, e4m3_values, moe_dense, unpack_matrix_nvfp4
from w4a16_group_quantized_moe_gb300 import inputs


def test_e2m1_matches_the_specification_table(oracle_mod):
    got = np.array([oracle_mod.e2m1_to_double(c) for c in range(16)])
    assert np.array_equal(got, E2M1_VALUES)
    assert np.array_equal(np.signbit(got), np.signbit(E2M1_VALUES))


def test_e4m3_matches_torch_for_every_byte(oracle_mod):
    ref = e4m3_values()
    got = np.array([oracle_mod.e4m3_to_double(b) for b in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(got))
    assert np.array_equal(got[~nan], ref[~nan])
    # anchors of the format: largest finite value, one, smallest normal and subnormal
    assert got[0x7E] == 448.0 and got[0x38] == 1.0 and got[0x08] == 2.0 ** -6 and got[0x01] == 2.0 ** -9


def _one_row(word, scale_bytes, gs, K=32, N=1, E=1):
    codes = np.zeros((E, N, K // 8), np.uint32)
    codes[0, 0, 0] = word
    bs = np.zeros((E, N, K // 16), np.uint8)
    bs[0, 0, :len(scale_bytes)] = scale_bytes
    return codes, bs, np.full(E, gs, np.float32)


def test_dequant_hand_derived_word(oracle_mod):
    # word 0x7A93_1F20: nibbles (kk 0..7) = 0, 2, 15, 1, 3, 9, 10, 7
    #   E2M1: 0, 1.0, -6.0, 0.5, 1.5, -0.5, -1.0, 6.0
    # block scale 0x40 = 2.0 (first 16 elements), per-expert scale 0.25
    w = _one_row(0x7A931F20, [0x40, 0x38], 0.25)
    want = [0.0, 1.0, -6.0, 0.5, 1.5, -0.5, -1.0, 6.0]
    for kk in range(8):
        assert oracle_mod.dequant_nvfp4(w, 1, 32, 0, 0, kk) == want[kk] * 2.0 * 0.25


def test_dequant_uses_the_block_of_sixteen(oracle_mod):
    # element 16 reads the second block scale (0x38 = 1.0), element 15 the first (0x40 = 2.0)
    codes = np.full((1, 1, 4), 0x22222222, np.uint32)   # every code 2 -> 1.0
    bs = np.array([[[0x40, 0x38]]], np.uint8)
    w = (codes, bs, np.ones(1, np.float32))
    assert oracle_mod.dequant_nvfp4(w, 1, 32, 0, 0, 15) == 2.0
    assert oracle_mod.dequant_nvfp4(w, 1, 32, 0, 0, 16) == 1.0


SHAPES = [inputs.MoEShape(3, 64, 32, 6, 2), inputs.MoEShape(2, 96, 64, 5, 3)]


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: f"T{s.T}H{s.H}I{s.I}")
def test_layer_matches_dense_brute_force(oracle_mod, sh):
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=5)
    w13, w2 = inputs.make_weights_nvfp4(sh.E, sh.H, sh.I, seed=5)
    ref = oracle_mod.moe_forward_nvfp4(logits, x, w13, w2, sh.k)
    out, _, _, ids, _ = moe_dense(logits, x, w13, w2, sh.k, unpack=unpack_matrix_nvfp4)
    assert np.array_equal(ref["topk_ids"], ids)
    np.testing.assert_allclose(ref["out"], out, rtol=1e-12, atol=1e-14)
    for t in range(sh.T):
        np.testing.assert_allclose(oracle_mod.moe_token_nvfp4(t, logits, x, w13, w2, sh.k), out[t],
                                   rtol=1e-12, atol=1e-14)


def test_layer_constant_closed_form(oracle_mod):
    # every weight e2m1(2) * e4m3(0x38) * c = c, every activation a:
    # g = u = H a c, h = silu(g) g, y = I h c, weights sum to one -> out = y
    E, H, I, k, T = 4, 64, 32, 2, 2
    c, a = 0.0625, 0.5
    codes13 = np.full((E, 2 * I, H // 8), 0x22222222, np.uint32)
    codes2 = np.full((E, H, I // 8), 0x22222222, np.uint32)
    w13 = (codes13, np.full((E, 2 * I, H // 16), 0x38, np.uint8), np.full(E, c, np.float32))
    w2 = (codes2, np.full((E, H, I // 16), 0x38, np.uint8), np.full(E, c, np.float32))
    logits = np.arange(T * E, dtype=np.float32).reshape(T, E)
    x = np.full((T, H), a, np.float16)
    g = H * a * c
    h = g / (1.0 + np.exp(-g)) * g
    y = I * h * c
    ref = oracle_mod.moe_forward_nvfp4(logits, x, w13, w2, k)
    np.testing.assert_allclose(ref["h"], h, rtol=1e-14)
    np.testing.assert_allclose(ref["out"], y, rtol=1e-13)


def test_h_of_the_grouped_step_matches_dense(oracle_mod):
    sh = SHAPES[0]
    logits, x = inputs.make_activations(sh.T, sh.H, sh.E, seed=8)
    w13, w2 = inputs.make_weights_nvfp4(sh.E, sh.H, sh.I, seed=8)
    ids, _ = oracle_mod.route(logits, sh.k)
    meta = oracle_mod.align(ids, sh.E)
    h = oracle_mod.gate_up_silu_nvfp4(x, w13, meta, sh.k)
    _, h_dense, _, _, _ = moe_dense(logits, x, w13, w2, sh.k, unpack=unpack_matrix_nvfp4)
    offs, sp, act, na = meta
    for r, p in enumerate(sp):
        e = int(ids.reshape(-1)[p])
        np.testing.assert_allclose(h[r], h_dense[e, p // sh.k], rtol=1e-12, atol=1e-14)
