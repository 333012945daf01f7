"""libmoe_w4a16: the W4A16 group-32 routed-expert MoE layer on GB300.

A thin binding over the C ABI in include/moe_w4a16.h.  The functions below
have the C names, take PyTorch CUDA tensors (PyTorch only provides device
memory and streams), and do argument marshalling only: every step of the
layer runs in the library's CUDA kernels.  There is no fallback path: if the
native library is missing the calls raise.

Build the library with ``python -m w4a16_group_quantized_moe_gb300.build``
(or ``__graft_entry__.build()``).
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_native", "libmoe_w4a16.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE_FLAG = 5

MOE_DEVERR_BAD_EXPERT_ID = 0x1
MOE_DEVERR_WAIT_TIMEOUT = 0x2
MOE_DEVERR_BAD_METADATA = 0x4

# diagnostic words of the workspace control block (u32 word indices)
MOE_CTRL_WAIT_POLLS = 1
MOE_CTRL_WAIT_EXTRA = 2
MOE_CTRL_TIMELINE = 4

MOE_PATH_NONE = 0
MOE_PATH_DECODE = 1
MOE_PATH_TENSOR_CORE = 2
MOE_PATH_STREAM = 3
MOE_PATH_AUTO = 0  # as an argument: the library's choice

EXPORTED = ("moe_abi_version", "moe_status_string", "moe_workspace_bytes", "moe_step_kernel_path",
            "moe_get_device_error", "moe_topk_route", "moe_align_offsets", "moe_topk_route_align",
            "moe_w4a16_gate_up_silu", "moe_w4a16_down_combine",
            "moe_w4a16_down_combine_noalloc", "moe_layer_workspace_bytes", "moe_w4a16_moe_layer",
            "moe_nvfp4_gate_up_silu", "moe_nvfp4_down_combine", "moe_nvfp4_moe_layer",
            "moe_router_logits", "moe_router_route_align", "moe_awq_import",
            "moe_w4a16_gate_up_silu_ex", "moe_w4a16_down_combine_ex", "moe_decode_layer_floor")

_lock = threading.Lock()
_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


class MoEError(RuntimeError):
    def __init__(self, call: str, status: int, text: str):
        super().__init__(f"{call} failed: {text} (status {status})")
        self.status = status


def load_library(path: str = LIB_PATH):
    """Loads libmoe_w4a16.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"libmoe_w4a16 native library not found at {path}; build it with "
                "`python -m w4a16_group_quantized_moe_gb300.build`")
        lib = ctypes.CDLL(path)
        lib.moe_abi_version.restype = _I
        lib.moe_status_string.restype = ctypes.c_char_p
        lib.moe_status_string.argtypes = [_I]
        lib.moe_workspace_bytes.restype = _SZ
        lib.moe_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
        lib.moe_step_kernel_path.restype = _I
        lib.moe_step_kernel_path.argtypes = [_I, _I, _I, _I, _I]
        lib.moe_get_device_error.restype = _I
        lib.moe_get_device_error.argtypes = [_P, _SZ, ctypes.POINTER(ctypes.c_uint32), _P]
        lib.moe_topk_route.restype = _I
        lib.moe_topk_route.argtypes = [_P, _I, _I, _I, _P, _P, _P]
        lib.moe_align_offsets.restype = _I
        lib.moe_align_offsets.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _SZ, _P]
        lib.moe_topk_route_align.restype = _I
        lib.moe_topk_route_align.argtypes = [_P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _SZ, _P]
        lib.moe_w4a16_gate_up_silu.restype = _I
        lib.moe_w4a16_gate_up_silu.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P,
                                               _I, _I, _I, _I, _I, _P, _P, _SZ, _P]
        lib.moe_w4a16_down_combine.restype = _I
        lib.moe_w4a16_down_combine.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                                               _I, _I, _I, _I, _I, _P, _P, _SZ, _P]
        lib.moe_w4a16_gate_up_silu_ex.restype = _I
        lib.moe_w4a16_gate_up_silu_ex.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P,
                                                  _I, _I, _I, _I, _I, _P, _P, _SZ, _I, _P]
        lib.moe_w4a16_down_combine_ex.restype = _I
        lib.moe_w4a16_down_combine_ex.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                                                  _I, _I, _I, _I, _I, _P, _P, _SZ, _I, _P]
        lib.moe_w4a16_down_combine_noalloc.restype = _I
        lib.moe_w4a16_down_combine_noalloc.argtypes = [_P, _P, _P, _P, _I, _P, _P, _P, _P, _P,
                                                       _I, _I, _I, _I, _I, _P, _P]
        lib.moe_decode_layer_floor.restype = _I
        lib.moe_decode_layer_floor.argtypes = [_I, _I, _I, _I, _I, _P]
        lib.moe_layer_workspace_bytes.restype = _SZ
        lib.moe_layer_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
        lib.moe_w4a16_moe_layer.restype = _I
        lib.moe_w4a16_moe_layer.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I,
                                            _P, _P, _P, _P, _SZ, _P]
        lib.moe_nvfp4_gate_up_silu.restype = _I
        lib.moe_nvfp4_gate_up_silu.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P,
                                               _I, _I, _I, _I, _I, _P, _P, _SZ, _P]
        lib.moe_nvfp4_down_combine.restype = _I
        lib.moe_nvfp4_down_combine.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P,
                                               _I, _I, _I, _I, _I, _P, _P, _SZ, _P]
        lib.moe_nvfp4_moe_layer.restype = _I
        lib.moe_nvfp4_moe_layer.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I,
                                            _P, _P, _P, _P, _SZ, _P]
        lib.moe_router_logits.restype = _I
        lib.moe_router_logits.argtypes = [_P, _P, _I, _I, _I, _P, _P, _SZ, _P]
        lib.moe_router_route_align.restype = _I
        lib.moe_router_route_align.argtypes = [_P, _P, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                               _P, _SZ, _P]
        lib.moe_awq_import.restype = _I
        lib.moe_awq_import.argtypes = [_P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _I, _I, _P]
        _lib = lib
        return lib


def _check(call: str, status: int):
    if status != MOE_OK:
        raise MoEError(call, status, load_library().moe_status_string(status).decode())


def _dev(t, dtype, name):
    """Device address of a contiguous CUDA tensor of the given dtype."""
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _stream(stream):
    import torch
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def workspace_bytes(T: int, E: int, k: int, H: int, I: int) -> int:
    return int(load_library().moe_workspace_bytes(T, E, k, H, I))


def new_workspace(T: int, E: int, k: int, H: int, I: int, device="cuda"):
    """A zero-filled workspace of the size the library asks for."""
    import torch
    n = workspace_bytes(T, E, k, H, I)
    if n == 0:
        raise MoEError("moe_workspace_bytes", MOE_ERR_INVALID_ARG, "sizes rejected")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def layer_workspace_bytes(T: int, E: int, k: int, H: int, I: int) -> int:
    return int(load_library().moe_layer_workspace_bytes(T, E, k, H, I))


def new_layer_workspace(T: int, E: int, k: int, H: int, I: int, device="cuda"):
    """A zero-filled workspace for moe_w4a16_moe_layer (also large enough for
    every step call of the same shape)."""
    import torch
    n = layer_workspace_bytes(T, E, k, H, I)
    if n == 0:
        raise MoEError("moe_layer_workspace_bytes", MOE_ERR_INVALID_ARG, "sizes rejected")
    return torch.zeros(n, dtype=torch.uint8, device=device)


def set_diagnostics(workspace, wait_polls: int = 0, wait_extra: int = 0, timeline=None):
    """Writes the diagnostic words of a workspace's control block (stream
    ordered): the poll limit of cross-CTA waits (0: default), an amount added
    to every such wait's target (nonzero: the waits run out), and the device
    buffer (int64, 8 per CTA) the one-call decode layer fills with phase
    timestamps (None: off)."""
    import torch
    words = torch.zeros(6, dtype=torch.int32)
    words[MOE_CTRL_WAIT_POLLS] = int(wait_polls)
    words[MOE_CTRL_WAIT_EXTRA] = int(wait_extra)
    tl = 0 if timeline is None else _dev(timeline, torch.int64, "timeline")
    words[MOE_CTRL_TIMELINE:MOE_CTRL_TIMELINE + 2] = torch.tensor([tl], dtype=torch.int64).view(torch.int32)
    workspace[4:24].copy_(words.view(torch.uint8)[4:24], non_blocking=False)


def moe_step_kernel_path(T: int, E: int, k: int, H: int, I: int) -> int:
    """MOE_PATH_* of the kernels the step calls run for this shape."""
    return int(load_library().moe_step_kernel_path(T, E, k, H, I))


def moe_decode_layer_floor(T: int, E: int, k: int, H: int, I: int, stream=None, check: bool = True) -> int:
    """Launches the empty kernel with the one-call layer's launch shape (the
    launch-cost floor); returns the status (raises unless OK when check)."""
    st = int(load_library().moe_decode_layer_floor(T, E, k, H, I, _stream(stream)))
    if check:
        _check("moe_decode_layer_floor", st)
    return st


def moe_get_device_error(workspace, stream=None) -> int:
    """Synchronises the stream; returns (and clears) the device error word."""
    import torch
    flag = ctypes.c_uint32(0)
    st = load_library().moe_get_device_error(_dev(workspace, torch.uint8, "workspace"),
                                             workspace.numel(), ctypes.byref(flag), _stream(stream))
    if st not in (MOE_OK, MOE_ERR_DEVICE_FLAG):
        _check("moe_get_device_error", st)
    return int(flag.value)


def moe_topk_route(logits, k: int, topk_ids=None, topk_w=None, stream=None):
    import torch
    T, E = logits.shape
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    _check("moe_topk_route", load_library().moe_topk_route(
        _dev(logits, torch.float32, "logits"), T, E, k, _dev(topk_ids, torch.int32, "topk_ids"),
        _dev(topk_w, torch.float32, "topk_w"), _stream(stream)))
    return topk_ids, topk_w


def moe_align_offsets(topk_ids, E: int, workspace=None, out=None, stream=None):
    """Returns (expert_offsets[E+1], sorted_pair[P], active_experts[E], num_active[1])."""
    import torch
    T, k = topk_ids.shape
    dev = topk_ids.device
    if out is None:
        out = (torch.empty(E + 1, dtype=torch.int32, device=dev),
               torch.empty(T * k, dtype=torch.int32, device=dev),
               torch.empty(E, dtype=torch.int32, device=dev),
               torch.empty(1, dtype=torch.int32, device=dev))
    offs, sp, act, na = out
    ws = _dev(workspace, torch.uint8, "workspace")
    _check("moe_align_offsets", load_library().moe_align_offsets(
        _dev(topk_ids, torch.int32, "topk_ids"), T, E, k, _dev(offs, torch.int32, "expert_offsets"),
        _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
        _dev(na, torch.int32, "num_active"), ws, 0 if workspace is None else workspace.numel(),
        _stream(stream)))
    return out


def moe_topk_route_align(logits, k: int, workspace=None, topk_ids=None, topk_w=None, meta=None,
                         stream=None):
    """Steps 1 and 2 in one call: (topk_ids, topk_w, meta)."""
    import torch
    T, E = logits.shape
    dev = logits.device
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if meta is None:
        meta = (torch.empty(E + 1, dtype=torch.int32, device=dev),
                torch.empty(T * k, dtype=torch.int32, device=dev),
                torch.empty(E, dtype=torch.int32, device=dev),
                torch.empty(1, dtype=torch.int32, device=dev))
    offs, sp, act, na = meta
    _check("moe_topk_route_align", load_library().moe_topk_route_align(
        _dev(logits, torch.float32, "logits"), T, E, k, _dev(topk_ids, torch.int32, "topk_ids"),
        _dev(topk_w, torch.float32, "topk_w"), _dev(offs, torch.int32, "expert_offsets"),
        _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
        _dev(na, torch.int32, "num_active"), _dev(workspace, torch.uint8, "workspace"),
        0 if workspace is None else workspace.numel(), _stream(stream)))
    return topk_ids, topk_w, meta


def moe_w4a16_gate_up_silu(x, w13, meta, k: int, workspace, h=None, stream=None, group_size=32,
                           path=MOE_PATH_AUTO):
    """h[T*k, I] (fp16, sorted-row order).  w13 = (qweight, scales, qzeros);
    path forces a kernel family (MOE_PATH_*; AUTO: the library's choice)."""
    import torch
    q, s, z = w13
    T, H = x.shape
    E, twoI, _ = q.shape
    I = twoI // 2
    offs, sp, act, na = meta
    if h is None:
        h = torch.empty((T * k, I), dtype=torch.float16, device=x.device)
    lib = load_library()
    args = (_dev(x, torch.float16, "x"), _dev(q, torch.int32, "w13_q"), _dev(s, torch.float16, "w13_s"),
            _dev(z, torch.int32, "w13_z"), group_size, _dev(offs, torch.int32, "expert_offsets"),
            _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
            _dev(na, torch.int32, "num_active"), T, E, k, H, I, _dev(h, torch.float16, "h"),
            _dev(workspace, torch.uint8, "workspace"), workspace.numel())
    if path == MOE_PATH_AUTO:
        _check("moe_w4a16_gate_up_silu", lib.moe_w4a16_gate_up_silu(*args, _stream(stream)))
    else:
        _check("moe_w4a16_gate_up_silu_ex", lib.moe_w4a16_gate_up_silu_ex(*args, path, _stream(stream)))
    return h


def moe_w4a16_down_combine(h, w2, meta, topk_w, workspace, out=None, stream=None, group_size=32,
                           path=MOE_PATH_AUTO):
    """out[T, H] (fp16).  w2 = (qweight, scales, qzeros); path as for
    moe_w4a16_gate_up_silu."""
    import torch
    q, s, z = w2
    E, H, _ = q.shape
    T, k = topk_w.shape
    I = h.shape[1]
    offs, sp, act, na = meta
    if out is None:
        out = torch.empty((T, H), dtype=torch.float16, device=h.device)
    lib = load_library()
    args = (_dev(h, torch.float16, "h"), _dev(q, torch.int32, "w2_q"), _dev(s, torch.float16, "w2_s"),
            _dev(z, torch.int32, "w2_z"), group_size, _dev(offs, torch.int32, "expert_offsets"),
            _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
            _dev(na, torch.int32, "num_active"), _dev(topk_w, torch.float32, "topk_w"),
            T, E, k, H, I, _dev(out, torch.float16, "out"),
            _dev(workspace, torch.uint8, "workspace"), workspace.numel())
    if path == MOE_PATH_AUTO:
        _check("moe_w4a16_down_combine", lib.moe_w4a16_down_combine(*args, _stream(stream)))
    else:
        _check("moe_w4a16_down_combine_ex", lib.moe_w4a16_down_combine_ex(*args, path, _stream(stream)))
    return out


def moe_w4a16_down_combine_noalloc(h, w2, meta, topk_w, out=None, stream=None, group_size=32):
    """out[T, H] (fp16) like moe_w4a16_down_combine, for callers that cannot
    allocate a workspace: the library's own fixed scratch array is used
    instead (see include/moe_w4a16.h; calls that overlap on the GPU race)."""
    import torch
    q, s, z = w2
    E, H, _ = q.shape
    T, k = topk_w.shape
    I = h.shape[1]
    offs, sp, act, na = meta
    if out is None:
        out = torch.empty((T, H), dtype=torch.float16, device=h.device)
    _check("moe_w4a16_down_combine_noalloc", load_library().moe_w4a16_down_combine_noalloc(
        _dev(h, torch.float16, "h"), _dev(q, torch.int32, "w2_q"), _dev(s, torch.float16, "w2_s"),
        _dev(z, torch.int32, "w2_z"), group_size, _dev(offs, torch.int32, "expert_offsets"),
        _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
        _dev(na, torch.int32, "num_active"), _dev(topk_w, torch.float32, "topk_w"),
        T, E, k, H, I, _dev(out, torch.float16, "out"), _stream(stream)))
    return out


def moe_w4a16_moe_layer(logits, x, w13, w2, k: int, workspace, topk_ids=None, topk_w=None,
                        out=None, stream=None, group_size=32):
    """The whole layer in one C call; returns (out, topk_ids, topk_w)."""
    import torch
    T, E = logits.shape
    H = x.shape[1]
    I = w2[0].shape[2] * 8
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float16, device=logits.device)
    q13, s13, z13 = w13
    q2, s2, z2 = w2
    st = load_library().moe_w4a16_moe_layer(
        _dev(logits, torch.float32, "logits"), _dev(x, torch.float16, "x"),
        _dev(q13, torch.int32, "w13_q"), _dev(s13, torch.float16, "w13_s"), _dev(z13, torch.int32, "w13_z"),
        _dev(q2, torch.int32, "w2_q"), _dev(s2, torch.float16, "w2_s"), _dev(z2, torch.int32, "w2_z"),
        group_size, T, E, k, H, I, _dev(topk_ids, torch.int32, "topk_ids"),
        _dev(topk_w, torch.float32, "topk_w"), _dev(out, torch.float16, "out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream))
    _check("moe_w4a16_moe_layer", st)
    return out, topk_ids, topk_w


def moe_nvfp4_gate_up_silu(x, w13, meta, k: int, workspace, h=None, stream=None):
    """h[T*k, I] (fp16, sorted-row order).  w13 = (codes, bscale, gscale) NVFP4."""
    import torch
    c, b, g = w13
    T, H = x.shape
    E, twoI, _ = c.shape
    I = twoI // 2
    offs, sp, act, na = meta
    if h is None:
        h = torch.empty((T * k, I), dtype=torch.float16, device=x.device)
    _check("moe_nvfp4_gate_up_silu", load_library().moe_nvfp4_gate_up_silu(
        _dev(x, torch.float16, "x"), _dev(c, torch.int32, "w13_codes"), _dev(b, torch.uint8, "w13_bscale"),
        _dev(g, torch.float32, "w13_gscale"), _dev(offs, torch.int32, "expert_offsets"),
        _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
        _dev(na, torch.int32, "num_active"), T, E, k, H, I, _dev(h, torch.float16, "h"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))
    return h


def moe_nvfp4_down_combine(h, w2, meta, topk_w, workspace, out=None, stream=None):
    """out[T, H] (fp16).  w2 = (codes, bscale, gscale) NVFP4."""
    import torch
    c, b, g = w2
    E, H, _ = c.shape
    T, k = topk_w.shape
    I = h.shape[1]
    offs, sp, act, na = meta
    if out is None:
        out = torch.empty((T, H), dtype=torch.float16, device=h.device)
    _check("moe_nvfp4_down_combine", load_library().moe_nvfp4_down_combine(
        _dev(h, torch.float16, "h"), _dev(c, torch.int32, "w2_codes"), _dev(b, torch.uint8, "w2_bscale"),
        _dev(g, torch.float32, "w2_gscale"), _dev(offs, torch.int32, "expert_offsets"),
        _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
        _dev(na, torch.int32, "num_active"), _dev(topk_w, torch.float32, "topk_w"),
        T, E, k, H, I, _dev(out, torch.float16, "out"),
        _dev(workspace, torch.uint8, "workspace"), workspace.numel(), _stream(stream)))
    return out


def moe_nvfp4_moe_layer(logits, x, w13, w2, k: int, workspace, topk_ids=None, topk_w=None,
                        out=None, stream=None):
    """The whole layer with NVFP4 weights in one C call; (out, topk_ids, topk_w)."""
    import torch
    T, E = logits.shape
    H = x.shape[1]
    I = w2[0].shape[2] * 8
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=logits.device)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=logits.device)
    if out is None:
        out = torch.empty((T, H), dtype=torch.float16, device=logits.device)
    c13, b13, g13 = w13
    c2, b2, g2 = w2
    _check("moe_nvfp4_moe_layer", load_library().moe_nvfp4_moe_layer(
        _dev(logits, torch.float32, "logits"), _dev(x, torch.float16, "x"),
        _dev(c13, torch.int32, "w13_codes"), _dev(b13, torch.uint8, "w13_bscale"),
        _dev(g13, torch.float32, "w13_gscale"), _dev(c2, torch.int32, "w2_codes"),
        _dev(b2, torch.uint8, "w2_bscale"), _dev(g2, torch.float32, "w2_gscale"),
        T, E, k, H, I, _dev(topk_ids, torch.int32, "topk_ids"), _dev(topk_w, torch.float32, "topk_w"),
        _dev(out, torch.float16, "out"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))
    return out, topk_ids, topk_w


def moe_router_logits(x, w_router, logits=None, workspace=None, stream=None):
    """logits [T, E] (fp32) = x [T, H] (fp16) times w_router [E, H] (fp16) transposed."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    if w_router.shape[1] != H:
        raise ValueError("w_router must be [E, H]")
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=x.device)
    ws = _dev(workspace, torch.uint8, "workspace") if workspace is not None else None
    _check("moe_router_logits", load_library().moe_router_logits(
        _dev(x, torch.float16, "x"), _dev(w_router, torch.float16, "w_router"), T, E, H,
        _dev(logits, torch.float32, "logits"), ws, workspace.numel() if workspace is not None else 0,
        _stream(stream)))
    return logits


def moe_router_route_align(x, w_router, k: int, workspace, logits=None, topk_ids=None, topk_w=None,
                           meta=None, stream=None):
    """Router logits, top-k routing and grouping in one call; returns
    (logits, topk_ids, topk_w, (offsets, sorted_pair, active, num_active))."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    dev = x.device
    if logits is None:
        logits = torch.empty((T, E), dtype=torch.float32, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
    if topk_w is None:
        topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
    if meta is None:
        meta = (torch.empty(E + 1, dtype=torch.int32, device=dev), torch.empty(T * k, dtype=torch.int32, device=dev),
                torch.empty(E, dtype=torch.int32, device=dev), torch.empty(1, dtype=torch.int32, device=dev))
    offs, sp, act, na = meta
    _check("moe_router_route_align", load_library().moe_router_route_align(
        _dev(x, torch.float16, "x"), _dev(w_router, torch.float16, "w_router"), T, E, k, H,
        _dev(logits, torch.float32, "logits"), _dev(topk_ids, torch.int32, "topk_ids"),
        _dev(topk_w, torch.float32, "topk_w"), _dev(offs, torch.int32, "expert_offsets"),
        _dev(sp, torch.int32, "sorted_pair"), _dev(act, torch.int32, "active_experts"),
        _dev(na, torch.int32, "num_active"), _dev(workspace, torch.uint8, "workspace"), workspace.numel(),
        _stream(stream)))
    return logits, topk_ids, topk_w, meta


def moe_awq_import(awq, dst, row0: int = 0, stream=None):
    """Repacks an AWQ GEMM-layout layer stack awq = (qweight [E][K][N/8],
    qzeros [E][K/32][N/8], scales [E][K/32][N]) into rows [row0, row0+N) of
    dst = (qweight [E][Ndst][K/8], scales [E][Ndst][K/32], qzeros
    [E][Ndst/8][K/32]), in place on the device; returns dst."""
    import torch
    aq, az, as_ = awq
    q, s, z = dst
    E, K, N8 = aq.shape
    Ndst = q.shape[1]
    if q.shape != (E, Ndst, K // 8) or s.shape != (E, Ndst, K // 32) or z.shape != (E, Ndst // 8, K // 32):
        raise ValueError("destination shapes do not match the AWQ layer")
    if az.shape != (E, K // 32, N8) or as_.shape != (E, K // 32, N8 * 8):
        raise ValueError("AWQ qzeros / scales shapes do not match qweight")
    _check("moe_awq_import", load_library().moe_awq_import(
        _dev(aq, torch.int32, "awq_qweight"), _dev(az, torch.int32, "awq_qzeros"),
        _dev(as_, torch.float16, "awq_scales"), E, K, N8 * 8, 32, _dev(q, torch.int32, "qweight"),
        _dev(s, torch.float16, "scales"), _dev(z, torch.int32, "qzeros"), Ndst, row0, _stream(stream)))
    return dst


def to_device_weights_nvfp4(w, device="cuda"):
    """(codes u32, bscale u8, gscale f32) numpy arrays -> CUDA tensors (codes viewed as int32)."""
    import numpy as np
    import torch
    c, b, g = w
    return (torch.from_numpy(np.ascontiguousarray(c).view(np.int32)).to(device),
            torch.from_numpy(np.ascontiguousarray(b)).to(device),
            torch.from_numpy(np.ascontiguousarray(g, dtype=np.float32)).to(device))


def to_device_weights(w, device="cuda"):
    """(qweight, scales, qzeros) numpy arrays -> CUDA tensors (u32 viewed as int32)."""
    import numpy as np
    import torch
    q, s, z = w
    return (torch.from_numpy(np.ascontiguousarray(q).view(np.int32)).to(device),
            torch.from_numpy(np.ascontiguousarray(s)).to(device),
            torch.from_numpy(np.ascontiguousarray(z).view(np.int32)).to(device))


class MoELayer:
    """Device weights plus preallocated buffers for one (T, E, k, H, I) shape;
    ``forward`` issues the four calls on one stream."""

    def __init__(self, w13, w2, T: int, k: int, device="cuda", path=MOE_PATH_AUTO):
        import torch
        self.w13, self.w2, self.path = w13, w2, path
        E, twoI, H8 = w13[0].shape
        self.E, self.I, self.H, self.T, self.k = E, twoI // 2, H8 * 8, T, k
        dev = torch.device(device)
        P = T * k
        self.topk_ids = torch.empty((T, k), dtype=torch.int32, device=dev)
        self.topk_w = torch.empty((T, k), dtype=torch.float32, device=dev)
        self.meta = (torch.empty(E + 1, dtype=torch.int32, device=dev),
                     torch.empty(P, dtype=torch.int32, device=dev),
                     torch.empty(E, dtype=torch.int32, device=dev),
                     torch.empty(1, dtype=torch.int32, device=dev))
        self.h = torch.empty((P, self.I), dtype=torch.float16, device=dev)
        self.out = torch.empty((T, self.H), dtype=torch.float16, device=dev)
        # sized for the one-call layer too (a superset of the step calls' needs)
        self.workspace = new_layer_workspace(T, E, k, self.H, self.I, device=dev)

    def forward(self, logits, x, stream=None):
        moe_topk_route(logits, self.k, self.topk_ids, self.topk_w, stream=stream)
        moe_align_offsets(self.topk_ids, self.E, self.workspace, out=self.meta, stream=stream)
        moe_w4a16_gate_up_silu(x, self.w13, self.meta, self.k, self.workspace, h=self.h,
                               stream=stream, path=self.path)
        moe_w4a16_down_combine(self.h, self.w2, self.meta, self.topk_w, self.workspace,
                               out=self.out, stream=stream, path=self.path)
        return self.out

    def forward_layer(self, logits, x, stream=None):
        """The same layer through the one-call entry point."""
        moe_w4a16_moe_layer(logits, x, self.w13, self.w2, self.k, self.workspace,
                            topk_ids=self.topk_ids, topk_w=self.topk_w, out=self.out, stream=stream)
        return self.out

    def bind(self, logits, x, stream=None):
        """Pre-marshals the four calls for fixed input buffers; returns four
        zero-argument callables (route, align, gate_up, down) that each make
        one C call, and sets self.route_align_call (steps 1-2 in one call) and
        self.layer_call (the whole layer through moe_w4a16_moe_layer).
        Used where host overhead must stay off the timeline."""
        import torch
        lib = load_library()
        st = _stream(stream)
        T, E, k, H, I = self.T, self.E, self.k, self.H, self.I
        offs, sp, act, na = (t.data_ptr() for t in self.meta)
        ws, wsb = self.workspace.data_ptr(), self.workspace.numel()
        _dev(logits, torch.float32, "logits")
        _dev(x, torch.float16, "x")
        q13, s13, z13 = (t.data_ptr() for t in self.w13)
        q2, s2, z2 = (t.data_ptr() for t in self.w2)
        a_route = (logits.data_ptr(), T, E, k, self.topk_ids.data_ptr(), self.topk_w.data_ptr(), st)
        a_align = (self.topk_ids.data_ptr(), T, E, k, offs, sp, act, na, ws, wsb, st)
        a_gu = (x.data_ptr(), q13, s13, z13, 32, offs, sp, act, na, T, E, k, H, I,
                self.h.data_ptr(), ws, wsb, st)
        a_dn = (self.h.data_ptr(), q2, s2, z2, 32, offs, sp, act, na, self.topk_w.data_ptr(),
                T, E, k, H, I, self.out.data_ptr(), ws, wsb, st)

        def call(fn, name, args):
            def run():
                status = fn(*args)
                if status != MOE_OK:
                    _check(name, status)
            return run
        a_ra = (logits.data_ptr(), T, E, k, self.topk_ids.data_ptr(), self.topk_w.data_ptr(),
                offs, sp, act, na, ws, wsb, st)
        self.route_align_call = call(lib.moe_topk_route_align, "moe_topk_route_align", a_ra)
        a_layer = (logits.data_ptr(), x.data_ptr(), q13, s13, z13, q2, s2, z2, 32, T, E, k, H, I,
                   self.topk_ids.data_ptr(), self.topk_w.data_ptr(), self.out.data_ptr(), ws, wsb, st)
        self.layer_call = call(lib.moe_w4a16_moe_layer, "moe_w4a16_moe_layer", a_layer)
        if self.path != MOE_PATH_AUTO:
            gu = call(lib.moe_w4a16_gate_up_silu_ex, "moe_w4a16_gate_up_silu_ex", a_gu[:-1] + (self.path, st))
            dn = call(lib.moe_w4a16_down_combine_ex, "moe_w4a16_down_combine_ex", a_dn[:-1] + (self.path, st))
        else:
            gu = call(lib.moe_w4a16_gate_up_silu, "moe_w4a16_gate_up_silu", a_gu)
            dn = call(lib.moe_w4a16_down_combine, "moe_w4a16_down_combine", a_dn)
        return (call(lib.moe_topk_route, "moe_topk_route", a_route),
                call(lib.moe_align_offsets, "moe_align_offsets", a_align), gu, dn)


class MoELayerNvfp4(MoELayer):
    """MoELayer with NVFP4 weights: w13 / w2 = (codes, bscale, gscale) CUDA
    tensors (to_device_weights_nvfp4); routing and grouping as for W4A16."""

    def forward(self, logits, x, stream=None):
        moe_topk_route(logits, self.k, self.topk_ids, self.topk_w, stream=stream)
        moe_align_offsets(self.topk_ids, self.E, self.workspace, out=self.meta, stream=stream)
        moe_nvfp4_gate_up_silu(x, self.w13, self.meta, self.k, self.workspace, h=self.h, stream=stream)
        moe_nvfp4_down_combine(self.h, self.w2, self.meta, self.topk_w, self.workspace,
                               out=self.out, stream=stream)
        return self.out

    def forward_layer(self, logits, x, stream=None):
        moe_nvfp4_moe_layer(logits, x, self.w13, self.w2, self.k, self.workspace,
                            topk_ids=self.topk_ids, topk_w=self.topk_w, out=self.out, stream=stream)
        return self.out

    def bind(self, logits, x, stream=None):
        """(route_align, gate_up, down) zero-argument callables, one C call
        each; sets self.layer_call (the whole layer in one call)."""
        import torch
        lib = load_library()
        st = _stream(stream)
        T, E, k, H, I = self.T, self.E, self.k, self.H, self.I
        offs, sp, act, na = (t.data_ptr() for t in self.meta)
        ws, wsb = self.workspace.data_ptr(), self.workspace.numel()
        _dev(logits, torch.float32, "logits")
        _dev(x, torch.float16, "x")
        c13, b13, g13 = (t.data_ptr() for t in self.w13)
        c2, b2, g2 = (t.data_ptr() for t in self.w2)

        def call(fn, name, args):
            def run():
                status = fn(*args)
                if status != MOE_OK:
                    _check(name, status)
            return run
        ra = call(lib.moe_topk_route_align, "moe_topk_route_align",
                  (logits.data_ptr(), T, E, k, self.topk_ids.data_ptr(), self.topk_w.data_ptr(),
                   offs, sp, act, na, ws, wsb, st))
        self.route_align_call = ra
        gu = call(lib.moe_nvfp4_gate_up_silu, "moe_nvfp4_gate_up_silu",
                  (x.data_ptr(), c13, b13, g13, offs, sp, act, na, T, E, k, H, I, self.h.data_ptr(),
                   ws, wsb, st))
        dn = call(lib.moe_nvfp4_down_combine, "moe_nvfp4_down_combine",
                  (self.h.data_ptr(), c2, b2, g2, offs, sp, act, na, self.topk_w.data_ptr(),
                   T, E, k, H, I, self.out.data_ptr(), ws, wsb, st))
        self.layer_call = call(lib.moe_nvfp4_moe_layer, "moe_nvfp4_moe_layer",
                               (logits.data_ptr(), x.data_ptr(), c13, b13, g13, c2, b2, g2, T, E, k, H, I,
                                self.topk_ids.data_ptr(), self.topk_w.data_ptr(), self.out.data_ptr(),
                                ws, wsb, st))
        return ra, gu, dn
