"""Programmatic dependent launch: the boundary kernels start while the
previous kernel on the stream finishes, and read nothing of global memory
before that kernel has completed ("mhc_boundary" page: the kernel's prologue
runs before griddepcontrol.wait). A producer kernel that lets its dependent
start at once and writes the residual only 20 us later stands in for the
layer kernel before the boundary; the boundary after it, eager and replayed
from a CUDA graph, must give bit for bit the results of a call on the
finished residual. Covers the slice-parallel decode and multi-item kernels,
the cluster kernel, and the unshifted forms (among them the collapse kernel
as a programmatic dependent of the coefficients kernel: pre-only up to 2048
tokens, unshifted up to 512)."""
import numpy as np
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
    ops.mhc_debug_set_pdl(1)


def _bits(t):
    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("form,T,H", [("shifted", 1, 7168), ("shifted", 64, 7168),
                                      ("shifted", 2048, 7168), ("shifted", 5, 512),
                                      ("unshifted", 8, 7168), ("unshifted", 300, 7168),
                                      ("unshifted", 700, 4096), ("pre", 1, 7168), ("pre", 512, 7168),
                                      ("pre", 1500, 4096)])
def test_boundary_after_a_late_producer(form, T, H):
    d = synth.make_inputs(T, H, seed=2000 + T + H)
    res_src = dev_bf16(d["residual"])
    res = torch.zeros_like(res_src)
    x, post, comb = dev_bf16(d["x"]), dev_f32(d["post"]), dev_f32(d["comb"])
    pl = dev_f32(d["pre_lag"]) if form == "shifted" else None
    scale, base, nw = dev_f32(d["scale"]), dev_f32(d["base"]), dev_f32(d["norm_w"])
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    ws = torch.empty(ops.workspace_bytes(T, H), dtype=torch.uint8, device="cuda")

    def outs():
        o = dict(layer_input=torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
                 pre_out=torch.empty(T, 4, device="cuda"), post_out=torch.empty(T, 4, device="cuda"),
                 comb_out=torch.empty(T, 4, 4, device="cuda"))
        if form != "pre":
            o["residual_out"] = torch.empty_like(res_src)
        return o

    def boundary(r, o, stream=None):
        if form == "pre":
            ops.mhc_pre(r, w, scale, base, nw, workspace=ws, stream=stream, **o)
        else:
            ops.mhc_boundary_fused(x, r, post, comb, w, scale, base, nw, pl, workspace=ws,
                                   stream=stream, **o)

    ref = outs()
    boundary(res_src, ref)
    torch.cuda.synchronize()

    def check(o, what):
        torch.cuda.synchronize()
        assert ops.mhc_get_device_status() == 0, what
        for k, v in ref.items():
            assert torch.equal(_bits(o[k]), _bits(v)), (what, k)

    # eager: producer, then the boundary on the buffer it writes
    got = outs()
    ops.mhc_debug_delayed_copy(res_src, res, 20_000)
    boundary(res, got)
    check(got, "eager")
    # captured pair, replayed twice with the buffer cleared in between
    got = outs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ops.mhc_debug_delayed_copy(res_src, res, 20_000, stream=s)
        boundary(res, got, stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            ops.mhc_debug_delayed_copy(res_src, res, 20_000, stream=s)
            boundary(res, got, stream=s)
    torch.cuda.synchronize()
    for rep in range(2):
        res.zero_()
        for v in got.values():
            v.zero_()
        torch.cuda.synchronize()
        g.replay()
        check(got, f"replay {rep}")
