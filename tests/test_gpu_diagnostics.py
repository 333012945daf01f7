"""Device-side error reporting, made to happen on purpose without faulting
anything: a cross-CTA wait of the one-launch decode layer that can never be
satisfied (its target raised through the workspace's diagnostic word) must
run out, report MOE_DEVERR_WAIT_TIMEOUT and return, leaving the context
usable; inconsistent grouping metadata planted on the host must be reported
as MOE_DEVERR_BAD_METADATA; and the phase timeline must be filled in order."""
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


def _close(got, ref):
    bound = TOL_REL * np.abs(ref).max() + TOL_ABS
    return np.abs(np.asarray(got, np.float64) - ref).max() <= bound


SHAPE = inputs.MoEShape(4, 512, 128, 64, 6)


def _layer(moe, sh, seed=3):
    logits, x, w13, w2 = inputs.make_workload(inputs.Workload("diag", sh), seed=seed)
    layer = moe.MoELayer(moe.to_device_weights(w13), moe.to_device_weights(w2), sh.T, sh.k)
    return layer, logits, x, w13, w2


def test_unsatisfiable_cross_cta_wait_times_out_and_the_context_survives(moe):
    layer, logits, x, w13, w2 = _layer(moe, SHAPE)
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    moe.set_diagnostics(layer.workspace, wait_polls=2000, wait_extra=1)
    layer.forward_layer(lg, xx)
    torch.cuda.synchronize()
    flag = moe.moe_get_device_error(layer.workspace)
    assert flag & moe.MOE_DEVERR_WAIT_TIMEOUT
    # a zeroed workspace restores normal operation on the same context
    layer.workspace.zero_()
    out = layer.forward_layer(lg, xx).float().cpu().numpy()
    assert moe.moe_get_device_error(layer.workspace) == 0
    assert _close(out, oracle.moe_forward(logits, x, w13, w2, SHAPE.k)["out"])


@pytest.mark.parametrize("sh,path", [(SHAPE, "MOE_PATH_DECODE"),
                                     (inputs.MoEShape(12, 2560, 640, 32, 10), "MOE_PATH_STREAM")],
                         ids=lambda v: f"T{v.T}" if hasattr(v, "T") else v)
def test_inconsistent_offsets_are_reported(moe, sh, path):
    """Bad offsets reach the gate/up kernels of the family named (forced
    through the _ex call) and are reported, not followed."""
    layer, logits, x, w13, w2 = _layer(moe, sh)
    ids, _ = oracle.route(logits, sh.k)
    offs, sp, act, na = oracle.align(ids, sh.E)
    bad = offs.copy()
    last = act[na - 1]
    bad[last + 1:] = sh.T * sh.k + 5          # the last segment ends past the pairs
    meta = (torch.from_numpy(bad).cuda(), torch.from_numpy(sp).cuda(), torch.from_numpy(act).cuda(),
            torch.tensor([na], dtype=torch.int32, device="cuda"))
    ws = moe.new_workspace(sh.T, sh.E, sh.k, sh.H, sh.I)
    moe.moe_w4a16_gate_up_silu(torch.from_numpy(x).cuda(), layer.w13, meta, sh.k, ws, path=getattr(moe, path))
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(ws) & moe.MOE_DEVERR_BAD_METADATA


def test_phase_timeline_is_filled_in_order(moe):
    layer, logits, x, w13, w2 = _layer(moe, SHAPE)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    tl = torch.zeros((n_sm, 8), dtype=torch.int64, device="cuda")
    moe.set_diagnostics(layer.workspace, timeline=tl)
    lg, xx = torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()
    layer.forward_layer(lg, xx)
    torch.cuda.synchronize()
    assert moe.moe_get_device_error(layer.workspace) == 0
    st = tl.cpu().numpy()
    entry, grouped, exitt = st[:, 0], st[:, 1], st[:, 7]
    assert np.all(entry > 0) and np.all(grouped >= entry) and np.all(exitt >= grouped)
    assert (exitt.max() - entry.min()) < 10_000_000   # one launch, well under 10 ms
    moe.set_diagnostics(layer.workspace)


def test_launch_floor_runs_where_the_one_launch_layer_does(moe):
    """The empty kernel with the layer's launch shape launches for decode
    shapes, is refused where the layer runs its four steps, and leaves the
    stream usable."""
    assert moe.moe_decode_layer_floor(1, 512, 10, 2560, 640) == moe.MOE_OK
    assert moe.moe_decode_layer_floor(4, SHAPE.E, SHAPE.k, SHAPE.H, SHAPE.I) == moe.MOE_OK
    assert moe.moe_decode_layer_floor(0, 512, 10, 2560, 640) == moe.MOE_OK
    assert moe.moe_decode_layer_floor(64, 512, 10, 2560, 640, check=False) == moe.MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    layer, logits, x, w13, w2 = _layer(moe, SHAPE)
    out = layer.forward_layer(torch.from_numpy(logits).cuda(), torch.from_numpy(x).cuda()).float().cpu().numpy()
    assert moe.moe_get_device_error(layer.workspace) == 0
    assert _close(out, oracle.moe_forward(logits, x, w13, w2, SHAPE.k)["out"])
