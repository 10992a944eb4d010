"""The allocation-free entry point, for callers that cannot allocate device
memory (an engine whose memory planner owns all device memory, or a loop
that cannot take cudaMalloc's implicit synchronisation): it must give the
same results as mhc_boundary_fused with a caller workspace, call after call,
while its scratch is the library's fixed device array.

Kept in a file of its own that pytest collects last. It passes run alone in
a fresh process and after the other tests."""
import ctypes

import numpy as np
import pytest
import torch

from manifold_constrained_hyper_gb300 import ops, synth

pytestmark = pytest.mark.gpu

F = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()
B = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from manifold_constrained_hyper_gb300 import build
    build.build()
    ops.load()


def _bits(t):
    return t.contiguous().view(torch.int32 if t.dtype == torch.float32 else torch.int16)


@pytest.mark.parametrize("T,H,shifted", [(64, 7168, True), (300, 1024, False), (5, 256, True)])
def test_noalloc_matches_workspace_entry_point_on_two_calls(T, H, shifted):
    d = synth.make_inputs(T, H, seed=900 + T)
    w = ops.mhc_prepare_weight(F(d["fn"]))
    x, res, post, comb = B(d["x"]), B(d["residual"]), F(d["post"]), F(d["comb"])
    scale, base, nw = F(d["scale"]), F(d["base"]), F(d["norm_w"])
    pl = F(d["pre_lag"]) if shifted else None
    ref = ops.mhc_boundary_fused(x, res, post, comb, w, scale, base, nw, pl)
    torch.cuda.synchronize()
    # outputs preallocated, so the second call allocates nothing at all
    outs = dict(residual_out=torch.empty_like(res),
                layer_input=torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
                pre_out=torch.empty(T, 4, device="cuda"),
                post_out=torch.empty(T, 4, device="cuda"),
                comb_out=torch.empty(T, 4, 4, device="cuda"))
    for call in range(2):
        for t in outs.values():
            t.view(torch.uint8).fill_(0xEE)          # stale values must be overwritten
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        got = ops.mhc_boundary_fused_noalloc(x, res, post, comb, w, scale, base, nw, pl, **outs)
        torch.cuda.synchronize()
        if call == 1:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert ops.mhc_get_device_status() == 0
        # same kernels, same order of every sum: bitwise equal to the workspace path
        for a, b in zip(got, ref):
            assert torch.equal(_bits(a), _bits(b)), f"call {call}"


@pytest.mark.parametrize("scratch", ["noalloc", "shared_workspace"])
def test_alternating_shapes_captured_and_eager_on_one_scratch(scratch):
    """Calls of two shapes (8 and 16 tokens at hidden 7168) share one scratch
    area: the library's fixed array, or one caller workspace sized for the
    larger. Each shape is captured into a CUDA graph of its own; replays of
    the two graphs are interleaved with eager calls of both shapes. A call's
    flag value must never be one that another shape's flag words already
    hold (a captured call takes its value from a cell at a fixed place of
    the scratch, never covered by any shape's flags); every output is
    compared bitwise with the workspace entry point on a private workspace."""
    H = 7168
    dev = "cuda"
    shapes = (8, 16)
    ws_shared = torch.empty(max(ops.workspace_bytes(T, H) for T in shapes), dtype=torch.uint8,
                            device=dev)
    case = {}
    for T in shapes:
        d = synth.make_inputs(T, H, seed=950 + T)
        c = dict(x=B(d["x"]), res=B(d["residual"]), post=F(d["post"]), comb=F(d["comb"]),
                 pl=F(d["pre_lag"]), w=ops.mhc_prepare_weight(F(d["fn"])), scale=F(d["scale"]),
                 base=F(d["base"]), nw=F(d["norm_w"]))
        c["ref"] = ops.mhc_boundary_fused(c["x"], c["res"], c["post"], c["comb"], c["w"],
                                          c["scale"], c["base"], c["nw"], c["pl"])
        c["outs"] = dict(residual_out=torch.empty_like(c["res"]),
                         layer_input=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                         pre_out=torch.empty(T, 4, device=dev), post_out=torch.empty(T, 4, device=dev),
                         comb_out=torch.empty(T, 4, 4, device=dev))
        case[T] = c
    torch.cuda.synchronize()

    def call(T, stream=None):
        c = case[T]
        args = (c["x"], c["res"], c["post"], c["comb"], c["w"], c["scale"], c["base"], c["nw"],
                c["pl"])
        if scratch == "noalloc":
            ops.mhc_boundary_fused_noalloc(*args, stream=stream, **c["outs"])
        else:
            ops.mhc_boundary_fused(*args, workspace=ws_shared, stream=stream, **c["outs"])

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graphs = {}
    with torch.cuda.stream(s):
        for T in shapes:
            call(T, stream=s)                        # first call on the device, before capture
        torch.cuda.synchronize()
        for T in shapes:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=s):
                call(T, stream=s)
            graphs[T] = g
    torch.cuda.synchronize()

    def check(T, what):
        torch.cuda.synchronize()
        assert ops.mhc_get_device_status() == 0, what
        for a, b in zip([case[T]["outs"][k] for k in ("residual_out", "layer_input", "pre_out",
                                                     "post_out", "comb_out")], case[T]["ref"]):
            assert torch.equal(_bits(a), _bits(b)), what
        for t in case[T]["outs"].values():
            t.view(torch.uint8).fill_(0xEE)
        torch.cuda.synchronize()

    for T in shapes:
        for t in case[T]["outs"].values():
            t.view(torch.uint8).fill_(0xEE)
    sequence = [("eager", 16), ("graph", 8), ("eager", 16), ("graph", 16), ("graph", 8),
                ("eager", 8), ("graph", 16), ("graph", 16), ("eager", 16), ("graph", 8),
                ("eager", 8), ("graph", 8), ("graph", 16)]
    for i, (kind, T) in enumerate(sequence):
        if kind == "eager":
            call(T)
        else:
            graphs[T].replay()
        check(T, f"step {i}: {kind} T={T}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = ops.load()
    p = ops.Params().c()
    A = ctypes.c_void_p(0x10000)                     # never dereferenced
    assert ops.workspace_bytes(4096, 7168) > 4 << 20
    rc = lib.mhc_boundary_fused_noalloc(A, A, A, A, A, A, A, A, None, 0, ctypes.byref(p), 4096,
                                        7168, A, A, A, A, A, None)
    assert rc == 8                                   # MHC_ERR_WORKSPACE, nothing enqueued
