"""Independent dense brute force of the MoE layer, in numpy float64.

Used only to pin the oracle.  It shares no code with the oracle: it unpacks
whole tensors with numpy bit operations, dequantises every expert densely,
takes the full softmax, ranks experts with a lexicographic sort, and evaluates
EVERY expert on EVERY token, with a gate that is zero outside the top-k.  This
is a different loop structure from the oracle's grouped evaluation (no
segments, no offsets, no sorted order).
"""
import numpy as np


def unpack_matrix(qweight, scales, qzeros):
    """Dense [E][N][K] float64 weights from the packed W4A16 g32 layout."""
    E, N, KW = qweight.shape
    K = KW * 8
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = (qweight[..., None] >> shifts) & np.uint32(0xF)          # [E][N][K/8][8]
    q = q.reshape(E, N, K).astype(np.float64)
    G = K // 32
    z = (qzeros[..., None] >> shifts) & np.uint32(0xF)           # [E][N/8][G][8]
    z = np.transpose(z, (0, 1, 3, 2)).reshape(E, N, G).astype(np.float64)
    s = np.asarray(scales, dtype=np.float16).astype(np.float64)  # [E][N][G]
    zf = np.repeat(z, 32, axis=2)
    sf = np.repeat(s, 32, axis=2)
    return (q - zf) * sf


# E2M1 values of the 16 codes (sign, 2 exponent bits, 1 mantissa bit), as
# tabulated in the OCP Microscaling Formats specification (FP4 E2M1).
E2M1_VALUES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0,
                        -0.0, -0.5, -1.0, -1.5, -2.0, -3.0, -4.0, -6.0])


def e4m3_values():
    """FP8 E4M3 value of each of the 256 bytes, decoded by PyTorch's
    float8_e4m3fn dtype (a library routine, not the oracle's decoder)."""
    import torch
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def unpack_matrix_nvfp4(codes, bscale, gscale):
    """Dense [E][N][K] float64 weights from the NVFP4 layout."""
    E, N, KW = codes.shape
    K = KW * 8
    shifts = (4 * np.arange(8, dtype=np.uint32))
    q = ((codes[..., None] >> shifts) & np.uint32(0xF)).reshape(E, N, K)
    v = E2M1_VALUES[q]
    bs = e4m3_values()[bscale]                                   # [E][N][K/16]
    return v * np.repeat(bs, 16, axis=2) * np.asarray(gscale, np.float64)[:, None, None]


def route_dense(logits, k):
    """Full softmax over E, rank by (logit desc, index asc), keep k, renormalise."""
    T, E = logits.shape
    lg = logits.astype(np.float64)
    p = np.exp(lg - lg.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ids = np.empty((T, k), np.int64)
    w = np.empty((T, k), np.float64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t].astype(np.float64)))
        ids[t] = order[:k]
        w[t] = p[t, ids[t]] / p[t, ids[t]].sum()
    return ids, w


def silu(v):
    return v / (1.0 + np.exp(-v))


def moe_dense(logits, x, w13, w2, k, unpack=unpack_matrix):
    """out [T][H], h_dense [E][T][I], gate [T][E] by dense evaluation."""
    W13 = unpack(*w13)                        # [E][2I][H]
    W2 = unpack(*w2)                          # [E][H][I]
    E, twoI, H = W13.shape
    I = twoI // 2
    T = logits.shape[0]
    xf = np.asarray(x, dtype=np.float16).astype(np.float64)
    ids, w = route_dense(logits, k)
    gate = np.zeros((T, E))
    for t in range(T):
        gate[t, ids[t]] = w[t]
    gu = np.einsum("th,enh->etn", xf, W13)    # [E][T][2I]
    h = silu(gu[..., :I]) * gu[..., I:]       # [E][T][I]
    y = np.einsum("eti,eni->etn", h, W2)      # [E][T][H]
    out = np.einsum("te,etn->tn", gate, y)
    return out, h, gate, ids, w
