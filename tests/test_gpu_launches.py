"""How many of the library's kernels one call launches, as counted by the
library itself (mhc_debug_launch_count): the shifted call is one kernel at
every size (the streaming kernel, or one thread-block cluster for a small
decode batch); an unshifted call of one tile in a single wave is one kernel
(its owner CTAs write the layer input), or two when the update is in place
(a collapse kernel follows); a longer unshifted call is three (streaming,
coefficients, collapse). The bench's gpu_launches is the same count over its
timed region."""
import pytest
import torch

from manifold_constrained_hyper_gb300 import ops, synth
from tests.mhc_testlib import dev_bf16, dev_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from manifold_constrained_hyper_gb300 import build
    build.build()
    ops.load()


def _count(call):
    torch.cuda.synchronize()
    n0 = ops.mhc_debug_launch_count()
    call()
    torch.cuda.synchronize()
    assert ops.mhc_get_device_status() == 0
    return ops.mhc_debug_launch_count() - n0


@pytest.mark.parametrize("form,T,H,in_place,expected",
                         [("shifted", 1, 7168, False, 1), ("shifted", 64, 7168, False, 1),
                          ("shifted", 1024, 7168, False, 1), ("shifted", 8, 512, False, 1),
                          ("unshifted", 1, 7168, False, 1), ("unshifted", 5, 7168, True, 2),
                          ("unshifted", 1024, 7168, False, 3), ("pre", 1, 7168, False, 1),
                          ("pre", 1024, 7168, False, 3)])
def test_kernels_per_call(form, T, H, in_place, expected):
    d = synth.make_inputs(T, H, seed=3100 + T + H)
    res = dev_bf16(d["residual"])
    x, post, comb, pl = dev_bf16(d["x"]), dev_f32(d["post"]), dev_f32(d["comb"]), dev_f32(d["pre_lag"])
    scale, base, nw = dev_f32(d["scale"]), dev_f32(d["base"]), dev_f32(d["norm_w"])
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    ws = torch.empty(ops.workspace_bytes(T, H), dtype=torch.uint8, device=res.device)
    if form == "pre":
        call = lambda: ops.mhc_pre(res, w, scale, base, nw, workspace=ws)
    else:
        kw = {"residual_out": res} if in_place else {}
        call = lambda: ops.mhc_boundary_fused(x, res, post, comb, w, scale, base, nw,
                                              pl if form == "shifted" else None,
                                              workspace=ws, **kw)
    call()                                  # first call: one-time set-up out of the count
    assert _count(call) == expected
    # the weight preparation is one kernel too
    assert _count(lambda: ops.mhc_prepare_weight(dev_f32(d["fn"]))) == 1
