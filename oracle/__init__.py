"""CPU oracle for the W4A16 group-32 routed-expert MoE layer.

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the benchmark's
CPU-baseline leg are the only users.  The product path (the CUDA library and
its Python binding) never imports this package.

The arithmetic lives in ``moe_oracle.c`` (plain C, IEEE double, single
thread); this module only compiles it with gcc and marshals numpy arrays.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle_moe.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile moe_oracle.c into a shared library (gcc, -O2, no fast-math)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.check_call([
        "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
        "-ffp-contract=off", "-fvisibility=hidden", "-Wall", "-Wextra",
        _SRC, "-o", tmp, "-lm",
    ])
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


_P = ctypes.c_void_p
_I = ctypes.c_int


def _declare(lib):
    lib.oracle_abi_version.restype = _I
    lib.oracle_half_to_double.restype = ctypes.c_double
    lib.oracle_half_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_dequant.restype = ctypes.c_double
    lib.oracle_dequant.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I]
    lib.oracle_route.argtypes = [_P, _I, _I, _I, _P, _P]
    lib.oracle_align.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P]
    lib.oracle_gate_up_silu.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P,
                                        _P, _P, _P, _P, _P]
    lib.oracle_down_combine.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P,
                                        _P, _P, _P, _P, _P, _P]
    lib.oracle_moe_token.argtypes = [_I, _P, _P, _I, _I, _I, _I,
                                     _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_moe_forward.argtypes = [_P, _P, _I, _I, _I, _I, _I,
                                       _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_e2m1_to_double.restype = ctypes.c_double
    lib.oracle_e2m1_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_double.restype = ctypes.c_double
    lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
    lib.oracle_dequant_nvfp4.restype = ctypes.c_double
    lib.oracle_dequant_nvfp4.argtypes = [_P, _P, _P, _I, _I, _I, _I, _I]
    lib.oracle_gate_up_silu_nvfp4.argtypes = [_P, _I, _I, _I, _I, _P, _P, _P,
                                              _P, _P, _P, _P, _P]
    lib.oracle_moe_token_nvfp4.argtypes = [_I, _P, _P, _I, _I, _I, _I,
                                           _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_moe_forward_nvfp4.argtypes = [_P, _P, _I, _I, _I, _I, _I,
                                             _P, _P, _P, _P, _P, _P,
                                             _P, _P, _P, _P, _P, _P, _P, _P]
    lib.oracle_router_logits.argtypes = [_P, _P, _I, _I, _I, _P]
    for f in (lib.oracle_awq_q, lib.oracle_awq_z):
        f.restype = _I
        f.argtypes = [_P, _I, _I, _I, _I, _I]
    lib.oracle_awq_s.restype = ctypes.c_uint16
    lib.oracle_awq_s.argtypes = [_P, _I, _I, _I, _I, _I]
    lib.oracle_awq_import.argtypes = [_P, _P, _P, _I, _I, _I, _P, _P, _P, _I, _I]
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


@contextlib.contextmanager
def using_library(path: str):
    """Run the wrappers against another build of the same C source (the pin
    tests use this to show that planted mistakes are caught)."""
    global _lib
    saved = _load()
    _lib = _declare(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = saved


def _c(a: np.ndarray, dtype) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.dtype(dtype):
        raise TypeError(f"expected {np.dtype(dtype)}, got {a.dtype}")
    return a


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def half_bits(a: np.ndarray) -> np.ndarray:
    """binary16 bit patterns of an fp16 array (no arithmetic)."""
    return np.ascontiguousarray(a, dtype=np.float16).view(np.uint16)


def half_to_double(bits: int) -> float:
    return _load().oracle_half_to_double(int(bits))


def dequant(qweight, scales, qzeros, N: int, K: int, e: int, n: int, kk: int) -> float:
    q = _c(qweight, np.uint32)
    s = half_bits(scales)
    z = _c(qzeros, np.uint32)
    return _load().oracle_dequant(_ptr(q), _ptr(s), _ptr(z), N, K, e, n, kk)


def route(logits: np.ndarray, k: int):
    lg = _c(logits, np.float32)
    T, E = lg.shape
    ids = np.empty((T, k), np.int32)
    w = np.empty((T, k), np.float64)
    _load().oracle_route(_ptr(lg), T, E, k, _ptr(ids), _ptr(w))
    return ids, w


def align(topk_ids: np.ndarray, E: int):
    ids = _c(topk_ids, np.int32)
    T, k = ids.shape
    offs = np.empty(E + 1, np.int32)
    sp = np.empty(T * k, np.int32)
    act = np.empty(E, np.int32)
    na = np.empty(1, np.int32)
    _load().oracle_align(_ptr(ids), T, E, k, _ptr(offs), _ptr(sp), _ptr(act), _ptr(na))
    return offs, sp, act, int(na[0])


def gate_up_silu(x, w13, meta, k: int):
    """h [T*k, I] (float64) in sorted-pair order.  meta = align(...) output."""
    xb = half_bits(x)
    T, H = xb.shape
    q, s, z = _c(w13[0], np.uint32), half_bits(w13[1]), _c(w13[2], np.uint32)
    I = q.shape[1] // 2
    offs, sp, act, na = meta
    na_arr = np.array([na], np.int32)
    h = np.zeros((T * k, I), np.float64)
    _load().oracle_gate_up_silu(_ptr(xb), T, H, I, k, _ptr(q), _ptr(s), _ptr(z),
                                _ptr(_c(offs, np.int32)), _ptr(_c(sp, np.int32)),
                                _ptr(_c(act, np.int32)), _ptr(na_arr), _ptr(h))
    return h


def down_combine(h, w2, meta, topk_w, T: int, k: int):
    hh = _c(h, np.float64)
    q, s, z = _c(w2[0], np.uint32), half_bits(w2[1]), _c(w2[2], np.uint32)
    H = q.shape[1]
    I = hh.shape[1]
    offs, sp, act, na = meta
    na_arr = np.array([na], np.int32)
    tw = _c(topk_w, np.float64)
    out = np.zeros((T, H), np.float64)
    _load().oracle_down_combine(_ptr(hh), T, H, I, k, _ptr(q), _ptr(s), _ptr(z),
                                _ptr(_c(offs, np.int32)), _ptr(_c(sp, np.int32)),
                                _ptr(_c(act, np.int32)), _ptr(na_arr), _ptr(tw),
                                _ptr(out))
    return out


def moe_token(t: int, logits, x, w13, w2, k: int) -> np.ndarray:
    """out[t] (float64 [H]) for one token, from the layer's definition."""
    lg = _c(logits, np.float32)
    xb = half_bits(x)
    E = lg.shape[1]
    H = xb.shape[1]
    q13, s13, z13 = _c(w13[0], np.uint32), half_bits(w13[1]), _c(w13[2], np.uint32)
    q2, s2, z2 = _c(w2[0], np.uint32), half_bits(w2[1]), _c(w2[2], np.uint32)
    I = q13.shape[1] // 2
    out = np.empty(H, np.float64)
    _load().oracle_moe_token(int(t), _ptr(lg), _ptr(xb), E, k, H, I,
                             _ptr(q13), _ptr(s13), _ptr(z13),
                             _ptr(q2), _ptr(s2), _ptr(z2), _ptr(out))
    return out


def moe_forward(logits, x, w13, w2, k: int) -> dict:
    """All four steps over a batch; returns every intermediate."""
    lg = _c(logits, np.float32)
    xb = half_bits(x)
    T, E = lg.shape
    H = xb.shape[1]
    q13, s13, z13 = _c(w13[0], np.uint32), half_bits(w13[1]), _c(w13[2], np.uint32)
    q2, s2, z2 = _c(w2[0], np.uint32), half_bits(w2[1]), _c(w2[2], np.uint32)
    I = q13.shape[1] // 2
    P = T * k
    r = dict(
        topk_ids=np.empty((T, k), np.int32), topk_w=np.empty((T, k), np.float64),
        expert_offsets=np.empty(E + 1, np.int32), sorted_pair=np.empty(P, np.int32),
        active_experts=np.empty(E, np.int32), num_active=np.empty(1, np.int32),
        h=np.zeros((P, I), np.float64), out=np.empty((T, H), np.float64),
    )
    _load().oracle_moe_forward(
        _ptr(lg), _ptr(xb), T, E, k, H, I, _ptr(q13), _ptr(s13), _ptr(z13),
        _ptr(q2), _ptr(s2), _ptr(z2), _ptr(r["topk_ids"]), _ptr(r["topk_w"]),
        _ptr(r["expert_offsets"]), _ptr(r["sorted_pair"]), _ptr(r["active_experts"]),
        _ptr(r["num_active"]), _ptr(r["h"]), _ptr(r["out"]))
    r["num_active"] = int(r["num_active"][0])
    return r


# ---------------------------------------------------------------- NVFP4
# Weights as (codes u32 [E][N][K/8], bscale u8 [E][N][K/16], gscale f32 [E]).

def e2m1_to_double(nib: int) -> float:
    return _load().oracle_e2m1_to_double(int(nib))


def e4m3_to_double(b: int) -> float:
    return _load().oracle_e4m3_to_double(int(b))


def _nv(w):
    return _c(w[0], np.uint32), _c(w[1], np.uint8), _c(w[2], np.float32)


def dequant_nvfp4(w, N: int, K: int, e: int, n: int, kk: int) -> float:
    c, b, g = _nv(w)
    return _load().oracle_dequant_nvfp4(_ptr(c), _ptr(b), _ptr(g), N, K, e, n, kk)


def gate_up_silu_nvfp4(x, w13, meta, k: int):
    """h [T*k, I] (float64) in sorted-pair order, NVFP4 gate/up weights."""
    xb = half_bits(x)
    T, H = xb.shape
    c, b, g = _nv(w13)
    I = c.shape[1] // 2
    offs, sp, act, na = meta
    na_arr = np.array([na], np.int32)
    h = np.zeros((T * k, I), np.float64)
    _load().oracle_gate_up_silu_nvfp4(_ptr(xb), T, H, I, k, _ptr(c), _ptr(b), _ptr(g),
                                      _ptr(_c(offs, np.int32)), _ptr(_c(sp, np.int32)),
                                      _ptr(_c(act, np.int32)), _ptr(na_arr), _ptr(h))
    return h


def moe_token_nvfp4(t: int, logits, x, w13, w2, k: int) -> np.ndarray:
    lg = _c(logits, np.float32)
    xb = half_bits(x)
    E = lg.shape[1]
    H = xb.shape[1]
    c13, b13, g13 = _nv(w13)
    c2, b2, g2 = _nv(w2)
    I = c13.shape[1] // 2
    out = np.empty(H, np.float64)
    _load().oracle_moe_token_nvfp4(int(t), _ptr(lg), _ptr(xb), E, k, H, I,
                                   _ptr(c13), _ptr(b13), _ptr(g13),
                                   _ptr(c2), _ptr(b2), _ptr(g2), _ptr(out))
    return out


def moe_forward_nvfp4(logits, x, w13, w2, k: int) -> dict:
    lg = _c(logits, np.float32)
    xb = half_bits(x)
    T, E = lg.shape
    H = xb.shape[1]
    c13, b13, g13 = _nv(w13)
    c2, b2, g2 = _nv(w2)
    I = c13.shape[1] // 2
    P = T * k
    r = dict(
        topk_ids=np.empty((T, k), np.int32), topk_w=np.empty((T, k), np.float64),
        expert_offsets=np.empty(E + 1, np.int32), sorted_pair=np.empty(P, np.int32),
        active_experts=np.empty(E, np.int32), num_active=np.empty(1, np.int32),
        h=np.zeros((P, I), np.float64), out=np.empty((T, H), np.float64),
    )
    _load().oracle_moe_forward_nvfp4(
        _ptr(lg), _ptr(xb), T, E, k, H, I, _ptr(c13), _ptr(b13), _ptr(g13),
        _ptr(c2), _ptr(b2), _ptr(g2), _ptr(r["topk_ids"]), _ptr(r["topk_w"]),
        _ptr(r["expert_offsets"]), _ptr(r["sorted_pair"]), _ptr(r["active_experts"]),
        _ptr(r["num_active"]), _ptr(r["h"]), _ptr(r["out"]))
    r["num_active"] = int(r["num_active"][0])
    return r


# ---------------------------------------------------------------- router logits
def router_logits(x, wr) -> np.ndarray:
    """logits [T, E] (float64) = x [T, H] (fp16) times wr [E, H] (fp16) transposed."""
    xb, wb = half_bits(x), half_bits(wr)
    T, H = xb.shape
    E = wb.shape[0]
    if wb.shape[1] != H:
        raise ValueError("router matrix must be [E, H]")
    out = np.empty((T, E), np.float64)
    _load().oracle_router_logits(_ptr(xb), _ptr(wb), T, E, H, _ptr(out))
    return out


# ---------------------------------------------------------------- AWQ import
# AWQ layer = (qweight u32 [E][K][N/8], qzeros u32 [E][K/32][N/8], scales f16 [E][K/32][N]).

def awq_element(awq, K: int, N: int, e: int, n: int, kk: int):
    """(q, z, scale bits) of element (n, kk) of expert e's AWQ layer."""
    aq, az, as_ = _c(awq[0], np.uint32), _c(awq[1], np.uint32), half_bits(awq[2])
    lib = _load()
    return (lib.oracle_awq_q(_ptr(aq), K, N, e, n, kk), lib.oracle_awq_z(_ptr(az), K, N, e, n, kk),
            lib.oracle_awq_s(_ptr(as_), K, N, e, n, kk))


def awq_import(awq, dst, row0: int = 0):
    """Writes the AWQ layer into rows [row0, row0+N) of dst = (qweight,
    scales, qzeros) in the layer's layout, in place; returns dst."""
    aq, az, as_ = _c(awq[0], np.uint32), _c(awq[1], np.uint32), half_bits(awq[2])
    E, K, N8 = aq.shape
    N = N8 * 8
    q, s, z = dst
    for a, dt in ((q, np.uint32), (z, np.uint32)):
        if a.dtype != dt or not a.flags.c_contiguous:
            raise TypeError("destination must be contiguous uint32")
    if s.dtype != np.float16 or not s.flags.c_contiguous:
        raise TypeError("destination scales must be contiguous float16")
    Ndst = q.shape[1]
    if q.shape != (E, Ndst, K // 8) or s.shape != (E, Ndst, K // 32) or z.shape != (E, Ndst // 8, K // 32):
        raise ValueError("destination shapes do not match")
    if row0 % 8 or row0 + N > Ndst:
        raise ValueError("row0 must be a multiple of 8 and the rows must fit")
    _load().oracle_awq_import(_ptr(aq), _ptr(az), _ptr(as_), E, K, N, _ptr(q), _ptr(s.view(np.uint16)),
                              _ptr(z), Ndst, row0)
    return dst
