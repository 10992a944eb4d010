"""Batch invariance (mhc_params.batch_invariant): a token's outputs do not
depend on the size of the batch it comes in or on its position in it, in
every form of the boundary and in the split-K pre. Checked bit for bit on
prefixes and a rotation of one seeded batch."""
import numpy as np
import pytest
import torch

from manifold_constrained_hyper_gb300 import ops, synth
from tests.mhc_testlib import dev_bf16, dev_f32

pytestmark = pytest.mark.gpu

INV = ops.Params(batch_invariant=True)


def _bits(t):
    return (t.view(torch.int16) if t.dtype == torch.bfloat16 else t).cpu().numpy()


def run_form(form, d, rows):
    res = dev_bf16(d["residual"][rows])
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    scale, base, nw = dev_f32(d["scale"]), dev_f32(d["base"]), dev_f32(d["norm_w"])
    if form == "pre":
        out = ops.mhc_pre(res, w, scale, base, nw, INV)
        names = ("layer_input", "pre", "post", "comb")
    elif form == "split_k":
        out = ops.mhc_pre_split_k(res, dev_f32(d["dot_mix"][:, rows]),
                                  dev_f32(d["sqrsum"][:, rows]), scale, base, nw, INV)
        names = ("layer_input", "pre", "post", "comb")
    else:
        pl = dev_f32(d["pre_lag"][rows]) if form == "shifted" else None
        out = ops.mhc_boundary_fused(dev_bf16(d["x"][rows]), res, dev_f32(d["post"][rows]),
                                     dev_f32(d["comb"][rows]), w, scale, base, nw, pl, INV)
        names = ("residual_out", "layer_input", "pre", "post", "comb")
    torch.cuda.synchronize()
    assert ops.mhc_get_device_status() == 0
    return {k: _bits(v) for k, v in zip(names, out)}


@pytest.mark.parametrize("form", ["shifted", "unshifted", "pre", "split_k"])
def test_outputs_do_not_depend_on_batch_size_or_position(form):
    T, H = 1100, 7168
    d = synth.make_split_k_inputs(T, H, 2, seed=880)
    full = run_form(form, d, np.arange(T))
    for n in (1, 3, 64, 129, 1024):
        part = run_form(form, d, np.arange(n))
        for k, v in part.items():
            assert np.array_equal(v, full[k][:n]), (form, n, k)
    perm = np.roll(np.arange(T), 37)
    rolled = run_form(form, d, perm)
    for k, v in rolled.items():
        assert np.array_equal(v, full[k][perm]), (form, "rolled", k)
