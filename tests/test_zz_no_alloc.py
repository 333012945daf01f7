"""The allocation-free down/combine entry point.

Some callers cannot call cudaMalloc (an engine that fixes its device memory
before serving, a plugin without access to the host's allocator), so the
library offers moe_w4a16_down_combine_noalloc, which keeps its scratch in a
fixed array inside the library instead of a caller workspace.  Here it is
called through the C ABI and must reproduce moe_w4a16_down_combine, twice in
a row (the shared array keeps the previous call's contents).  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest

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


# a decode batch (fused-combine kernels) and a larger one (staged kernels)
SHAPES = [inputs.MoEShape(4, 512, 128, 64, 6), inputs.MoEShape(12, 512, 128, 64, 6)]


@pytest.mark.parametrize("sh", SHAPES, ids=lambda s: f"T{s.T}")
def test_noalloc_matches_workspace_call_twice(moe, sh):
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("na", sh), seed=7)
    dw13, dw2 = moe.to_device_weights(w13), moe.to_device_weights(w2)
    layer = moe.MoELayer(dw13, dw2, sh.T, sh.k)
    ref = layer.forward(torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()).clone()
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(layer.workspace) == 0
    ref_np = ref.float().cpu().numpy()
    bound = TOL_REL * np.abs(ref_np).max() + TOL_ABS

    lib = moe.load_library()
    offs, sp, act, na = layer.meta
    stream = torch.cuda.current_stream().cuda_stream
    for call in range(2):
        out = torch.full((sh.T, sh.H), float("nan"), dtype=torch.float16, device="cuda")
        st = lib.moe_w4a16_down_combine_noalloc(
            layer.h.data_ptr(), dw2[0].data_ptr(), dw2[1].data_ptr(), dw2[2].data_ptr(), 32,
            offs.data_ptr(), sp.data_ptr(), act.data_ptr(), na.data_ptr(), layer.topk_w.data_ptr(),
            sh.T, sh.E, sh.k, sh.H, sh.I, out.data_ptr(), ctypes.c_void_p(stream))
        assert st == moe.MOE_OK, f"call {call}: status {st}"
        torch.cuda.synchronize()
        got = out.float().cpu().numpy()
        assert np.all(np.isfinite(got)), f"call {call}: non-finite output"
        err = np.abs(got - ref_np).max()
        assert err <= bound, f"call {call}: max err {err:.3e} > {bound:.3e}"


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
