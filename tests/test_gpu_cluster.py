"""The shifted boundary of decode batches on one thread-block cluster ("mhc_boundary"
page, MhcBoundaryKernel: the hidden slices of a token tile in one cluster,
partial mixes and sums of squares pushed over distributed shared memory and
summed in rank order), against the CPU oracle at the parity bar of the other
paths: residual_out bit-exact, layer input within 1 bf16 ulp, coefficients
within 1e-5 relative + 1e-7, mixes within 1e-5 of max(|mix|, ||terms||_2).
Also: both decode paths (cluster and slice-parallel) on the same inputs,
determinism, graph capture, the default path choice, and the shapes whose
cluster sizes are not powers of two. These tests force the cluster kernel
wherever it can run (by default it runs only where it is the faster path)."""
import numpy as np
import pytest
import torch

from manifold_constrained_hyper_gb300 import ops, synth
from tests.mhc_testlib import (bf16_ulp_diff, compare, dev_bf16, dev_f32, host_bits, run_gpu,
                               run_oracle)

pytestmark = pytest.mark.gpu

DISTINCT_SCALES = (0.25, 1.5, 3.0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from manifold_constrained_hyper_gb300 import build
    build.build()
    ops.load()
    ops.mhc_debug_set_decode_path(2)          # the cluster kernel wherever it can run
    yield
    ops.mhc_debug_set_decode_path(0)


@pytest.mark.parametrize("T", [1, 2, 4, 7, 8, 9, 16, 17, 31, 32, 33, 48, 63, 64])
def test_cluster_decode_sweep_h7168(T):
    """Every decode size at hidden 7168: a cluster of 16 CTAs, 14 chunks each
    (all resident up to 8 tokens, a ring of stages above)."""
    assert ops.plan_cluster(T, 7168) == 16
    d = synth.make_inputs(**synth.decode_workload(T))
    g = run_gpu("shifted", d)
    assert g["path"] == "cluster"
    compare("shifted", g, run_oracle("shifted", d))


@pytest.mark.parametrize("T,H,C", [(3, 32, 1), (5, 96, 3), (6, 160, 5), (4, 256, 8), (40, 256, 8),
                                   (12, 1024, 16), (64, 4096, 16), (2, 16384, 16), (64, 16384, 16),
                                   (9, 480, 15), (20, 224, 7)])
def test_cluster_shapes(T, H, C):
    """Cluster sizes from 1 to 16, odd ones included (H/32 = 3, 5, 7, 15
    chunks), and the most chunks per CTA (32 at hidden 16384)."""
    assert ops.plan_cluster(T, H) == C
    d = synth.make_inputs(T, H, seed=1300 + T + H)
    g = run_gpu("shifted", d)
    assert g["path"] == "cluster"
    compare("shifted", g, run_oracle("shifted", d))


@pytest.mark.parametrize("norm", ["bf16", None])
@pytest.mark.parametrize("T", [3, 40])
def test_cluster_norm_weight_variants(norm, T):
    d = synth.make_inputs(T, 7168, seed=1400 + T)
    g = run_gpu("shifted", d, norm=norm)
    compare("shifted", g, run_oracle("shifted", d, norm=norm))


@pytest.mark.parametrize("T", [1, 64])
def test_cluster_distinct_scales_and_saturation(T):
    """Distinct per-group scales, and stress-like values (outliers, base
    ~ N(0, 4) saturating the sigmoids) with 1 and 5 Sinkhorn iterations."""
    d = synth.make_inputs(T, 7168, seed=1500 + T, scale=DISTINCT_SCALES)
    compare("shifted", run_gpu("shifted", d), run_oracle("shifted", d))
    d = synth.make_inputs(T, 7168, seed=1510 + T, residual_std=8.0, outlier_frac=0.01,
                          outlier_mult=100.0, base_std=4.0)
    for iters in (1, 5):
        p = ops.Params(sinkhorn_iters=iters)
        compare("shifted", run_gpu("shifted", d, params=p), run_oracle("shifted", d, params=p))


def test_cluster_in_place_and_guarded_outputs():
    T, H = 9, 7168
    d = synth.make_inputs(T, H, seed=1600)
    o = run_oracle("shifted", d)
    g = run_gpu("shifted", d, in_place=True)
    compare("shifted", g, o)
    G = 4096
    canary = 0x5A5A
    big_res = torch.full((G * 2 + T * 4 * H,), canary, dtype=torch.int16, device="cuda")
    big_li = torch.full((G * 2 + T * H,), canary, dtype=torch.int16, device="cuda")
    big_f = torch.full((3, G * 2 + T * 16), 12345.0, device="cuda")
    rout = big_res[G:G + T * 4 * H].view(torch.bfloat16).view(T, 4, H)
    li = big_li[G:G + T * H].view(torch.bfloat16).view(T, H)
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    ops.mhc_boundary_fused(dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_f32(d["post"]),
                           dev_f32(d["comb"]), w, dev_f32(d["scale"]), dev_f32(d["base"]),
                           dev_f32(d["norm_w"]), dev_f32(d["pre_lag"]), residual_out=rout,
                           layer_input=li, pre_out=big_f[0, G:G + T * 4].view(T, 4),
                           post_out=big_f[1, G:G + T * 4].view(T, 4),
                           comb_out=big_f[2, G:G + T * 16].view(T, 4, 4))
    torch.cuda.synchronize()
    assert ops.mhc_get_device_status() == 0
    for big, n in ((big_res, T * 4 * H), (big_li, T * H)):
        assert torch.all(big[:G] == canary) and torch.all(big[G + n:] == canary)
    for i, n in enumerate((T * 4, T * 4, T * 16)):
        assert torch.all(big_f[i, :G] == 12345.0) and torch.all(big_f[i, G + n:] == 12345.0)
    assert np.array_equal(host_bits(rout), o["residual_out"])
    assert bf16_ulp_diff(host_bits(li), o["layer_input"]).max() <= 1


@pytest.mark.parametrize("T", [1, 8, 64])
def test_cluster_and_slice_paths_agree_and_are_deterministic(T):
    """The two decode paths on the same inputs: the residual bit for bit, the
    layer input within 1 ulp of each other (each within 1 ulp of the
    oracle), the coefficients within the parity bar; the cluster path is
    bitwise identical over 10 runs."""
    d = synth.make_inputs(T, 7168, seed=1700 + T)
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    runs = [run_gpu("shifted", d, weight=w) for _ in range(10)]
    assert all(r["path"] == "cluster" for r in runs)
    for r in runs[1:]:
        for k in ("residual_out_dev", "layer_input_dev"):
            assert torch.equal(r[k], runs[0][k]), k
        for k in ("pre", "post", "comb"):
            assert np.array_equal(r[k].view(np.uint32), runs[0][k].view(np.uint32)), k
    ops.mhc_debug_set_decode_path(1)
    try:
        s = run_gpu("shifted", d, weight=w)
    finally:
        ops.mhc_debug_set_decode_path(2)
    assert s["path"] == "slices" or ops.plan_cluster(T, 7168) == 0
    c = runs[0]
    assert torch.equal(c["residual_out_dev"], s["residual_out_dev"])
    assert bf16_ulp_diff(host_bits(c["layer_input_dev"]), host_bits(s["layer_input_dev"])).max() <= 1
    for k in ("pre", "post", "comb"):
        assert np.all(np.abs(c[k] - s[k]) <= 1e-5 * np.abs(s[k]) + 1e-7), k
    o = run_oracle("shifted", d)
    compare("shifted", s, o)
    compare("shifted", c, o)


@pytest.mark.parametrize("T", [1, 64])
def test_cluster_calls_capture_and_replay_with_new_inputs(T):
    """A captured cluster call replays with new inputs written into the same
    buffers and gives the eager results bit for bit (the call carries no
    per-call state: no flags, no epoch)."""
    H = 7168
    A = synth.make_inputs(T, H, seed=1800 + T)
    B = synth.make_inputs(T, H, seed=1801 + T)
    inp = {k: dev_bf16(A[k]) for k in ("residual", "x")} | \
          {k: dev_f32(A[k]) for k in ("post", "comb", "pre_lag")}
    scale, base, nw = dev_f32(A["scale"]), dev_f32(A["base"]), dev_f32(A["norm_w"])
    w = ops.mhc_prepare_weight(dev_f32(A["fn"]))
    outs = dict(residual_out=torch.empty_like(inp["residual"]),
                layer_input=torch.empty(T, H, dtype=torch.bfloat16, device="cuda"),
                pre_out=torch.empty(T, 4, device="cuda"), post_out=torch.empty(T, 4, device="cuda"),
                comb_out=torch.empty(T, 4, 4, device="cuda"))

    def call(stream=None):
        return ops.mhc_boundary_fused(inp["x"], inp["residual"], inp["post"], inp["comb"], w, scale,
                                      base, nw, inp["pre_lag"], stream=stream, **outs)

    def load(dd):
        for k in ("residual", "x"):
            inp[k].copy_(dev_bf16(dd[k]))
        for k in ("post", "comb", "pre_lag"):
            inp[k].copy_(dev_f32(dd[k]))

    load(B)
    eager = [t.clone() for t in call()]
    torch.cuda.synchronize()
    load(A)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(stream=s)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            call(stream=s)
    torch.cuda.synchronize()
    load(B)
    for t in outs.values():
        t.zero_()
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    assert ops.mhc_get_device_status() == 0
    got = [outs[k] for k in ("residual_out", "layer_input", "pre_out", "post_out", "comb_out")]
    for a_, b_ in zip(eager, got):
        if a_.dtype == torch.bfloat16:
            a_, b_ = a_.view(torch.int16), b_.view(torch.int16)
        assert torch.equal(a_, b_)


def test_default_path_choice():
    """By default the cluster kernel takes the shapes where it is the faster
    path: one chunk per CTA, two for up to 32 tokens, up to four for up to
    16 tokens."""
    ops.mhc_debug_set_decode_path(0)
    try:
        assert ops.plan_cluster(1, 256) == 8 and ops.plan_cluster(64, 512) == 16
        assert ops.plan_cluster(32, 1024) == 16 and ops.plan_cluster(33, 1024) == 0
        assert ops.plan_cluster(16, 2048) == 16 and ops.plan_cluster(17, 2048) == 0
        assert ops.plan_cluster(1, 4096) == 0 and ops.plan_cluster(1, 7168) == 0
        assert ops.plan_cluster(64, 4096) == 0
        for T, H, path in [(5, 512, "cluster"), (32, 1024, "cluster"), (16, 2048, "cluster"),
                           (17, 2048, "slices")]:
            d = synth.make_inputs(T, H, seed=1900 + T + H)
            g = run_gpu("shifted", d)
            assert g["path"] == path
            compare("shifted", g, run_oracle("shifted", d))
    finally:
        ops.mhc_debug_set_decode_path(2)
