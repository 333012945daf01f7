"""The allocation-free down/combine entry point.

Some callers cannot call cudaMalloc (an engine that fixes its device memory
before serving, a plugin without access to the host's allocator), so the
library offers moe_w4a16_down_combine_noalloc, which keeps its scratch in a
fixed array inside the library instead of a caller workspace.  Here it is
called through the C ABI, on every kernel path of the step, and must agree
with the oracle and with moe_w4a16_down_combine, twice in a row (the shared
array keeps the previous call's contents).  This file is collected last on
purpose."""
import ctypes

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


# Shapes inside the 8 MiB scratch on each family the automatic choice takes
# for the down/combine step: the decode kernels (fused combine; at 12 tokens
# on the full hidden size with h read from global memory) and the
# tensor-core kernels (per-pair projections in the scratch, then the combine
# kernel), the latter with fewer sorted rows than one 128-row chunk (P = 102)
# and with several chunks.
SHAPES = [
    (inputs.MoEShape(4, 512, 128, 64, 6), "MOE_PATH_DECODE"),
    (inputs.MoEShape(12, 2560, 640, 32, 10), "MOE_PATH_DECODE"),
    (inputs.MoEShape(17, 512, 128, 64, 6), "MOE_PATH_TENSOR_CORE"),
    (inputs.MoEShape(64, 512, 128, 16, 4), "MOE_PATH_TENSOR_CORE"),
]


def _oracle_step4_inputs(logits, x, w13, sh):
    """Routing, grouping and h from the oracle alone; h rounded to fp16 as
    the library stores it (the inputs of step 4)."""
    ids, tw = oracle.route(logits, sh.k)
    meta = oracle.align(ids, sh.E)
    h16 = oracle.gate_up_silu(x, w13, meta, sh.k).astype(np.float16)
    return ids, tw, meta, h16


@pytest.mark.parametrize("sh,path", SHAPES, ids=lambda v: f"T{v.T}" if hasattr(v, "T") else v)
def test_noalloc_matches_oracle_and_workspace_call_twice(moe, sh, path):
    assert moe.moe_step_kernel_path(sh.T, sh.E, sh.k, sh.H, sh.I) == getattr(moe, path)
    assert moe.workspace_bytes(sh.T, sh.E, sh.k, sh.H, sh.I) <= 8 << 20
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("na", sh), seed=7)
    ids, tw, meta, h16 = _oracle_step4_inputs(logits, x, w13, sh)
    ref_out = oracle.down_combine(h16.astype(np.float64), w2, meta, tw, sh.T, sh.k)
    bound = TOL_REL * np.abs(ref_out).max() + TOL_ABS

    dev = "cuda"
    dw2 = moe.to_device_weights(w2)
    d_h = torch.from_numpy(h16).to(dev)
    d_tw = torch.from_numpy(tw.astype(np.float32)).to(dev)
    offs, sp, act = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in meta[:3])
    na = torch.tensor([meta[3]], dtype=torch.int32, device=dev)
    d_meta = (offs, sp, act, na)

    # the existing entry point with a workspace, for comparison
    ws = moe.new_workspace(sh.T, sh.E, sh.k, sh.H, sh.I)
    ws_out = moe.moe_w4a16_down_combine(d_h, dw2, d_meta, d_tw, ws).float().cpu().numpy()
    assert moe.moe_get_device_error(ws) == 0

    lib = moe.load_library()
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((sh.T, sh.H), float("nan"), dtype=torch.float16, device=dev)
        st = lib.moe_w4a16_down_combine_noalloc(
            d_h.data_ptr(), dw2[0].data_ptr(), dw2[1].data_ptr(), dw2[2].data_ptr(), 32,
            offs.data_ptr(), sp.data_ptr(), act.data_ptr(), na.data_ptr(), d_tw.data_ptr(),
            sh.T, sh.E, sh.k, sh.H, sh.I, out.data_ptr(), ctypes.c_void_p(stream))
        assert st == moe.MOE_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        err = np.abs(got - ref_out).max()
        assert err <= bound, f"call {call}: max err vs oracle {err:.3e} > {bound:.3e}"
        err_ws = np.abs(got - ws_out).max()
        assert err_ws <= bound, f"call {call}: max err vs workspace call {err_ws:.3e} > {bound:.3e}"


def test_noalloc_rejects_shapes_beyond_its_scratch(moe):
    lib = moe.load_library()
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    p = buf.data_ptr()
    T, E, k, H, I = 2000, 64, 8, 512, 128      # needs ~33 MB of projections
    assert lib.moe_workspace_bytes(T, E, k, H, I) > 8 << 20
    st = lib.moe_w4a16_down_combine_noalloc(p, p, p, p, 32, p, p, p, p, p, T, E, k, H, I, p, None)
    assert st == moe.MOE_ERR_UNSUPPORTED
    st = lib.moe_w4a16_down_combine_noalloc(p, p, p, p, 32, p, p, p, p, p, 4, E, k, 500, I, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG        # H not a multiple of 32
    st = lib.moe_w4a16_down_combine_noalloc(p, p, p, p, 16, p, p, p, p, p, 4, E, k, H, I, p, None)
    assert st == moe.MOE_ERR_UNSUPPORTED        # group size other than 32
    st = lib.moe_w4a16_down_combine_noalloc(p + 4, p, p, p, 32, p, p, p, p, p, 4, E, k, H, I, p, None)
    assert st == moe.MOE_ERR_INVALID_ARG        # misaligned h
