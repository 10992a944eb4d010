"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs. Bar: bit-exact for the prepared weight and the updated
residual; layer input within 1 bf16 ulp (shifted, where the collapse is
exact) or 2 ulps (unshifted, where pre feeds a second bf16 rounding);
coefficients within 1e-5 relative + 1e-7; mixes within 1e-5 of
max(|mix|, ||terms||_2)."""
import numpy as np
import pytest
import torch

import oracle as orc
from manifold_constrained_hyper_gb300 import ops, synth
from tests.mhc_testlib import (bf16_ulp_diff, compare, dev_bf16, dev_f32, host_bits, run_gpu,
                               run_oracle)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from manifold_constrained_hyper_gb300 import build
    build.build()
    ops.load()


# ------------------------------------------------------------------ weight prep


@pytest.mark.parametrize("H", [32, 256, 4096, 7168])
def test_prepare_weight_bit_exact(H):
    d = synth.make_inputs(1, H, seed=100 + H)
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    torch.cuda.synchronize()
    got = w.cpu().numpy().view(np.uint16)
    assert np.array_equal(got, orc.weight_tiles(d["fn"], H))


def test_prepare_weight_rounding_edge_values():
    H = 32
    fn = np.zeros((24, 4 * H), np.float32)
    # ties, carries, signed zeros, a large value whose rounding carries into
    # the exponent, a tiny one, subnormals (weights whose TF32 rounding
    # overflows to inf are outside the finite-weight domain)
    special = np.array([0x3F801000, 0xBF801000, 0x3F800FFF, 0x3FFFF000, 0x00000000,
                        0x80000000, 0x7E7FF000, 0x33FFFFFF, 0x00001000, 0x80018000],
                       np.uint32).view(np.float32)
    fn.reshape(-1)[: special.size] = special
    fn.reshape(-1)[100:100 + 1000] = np.random.default_rng(1).standard_normal(1000)
    w = ops.mhc_prepare_weight(dev_f32(fn))
    torch.cuda.synchronize()
    assert np.array_equal(w.cpu().numpy().view(np.uint16), orc.weight_tiles(fn, H))


# ------------------------------------------------------------------ post


@pytest.mark.parametrize("T,H", [(1, 256), (3, 7168), (17, 512), (200, 4096)])
def test_post_bit_exact(T, H):
    d = synth.make_inputs(T, H, seed=200 + T)
    out = ops.mhc_post(dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_f32(d["post"]),
                       dev_f32(d["comb"]))
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(out), orc.post(d["x"], d["residual"], d["post"], d["comb"]))


def test_post_in_place_and_subnormals():
    T, H = 5, 256
    d = synth.make_inputs(T, H, seed=205)
    d["residual"][0, 0, :8] = np.array([1, 2, 0x8001, 0x0080, 0x007F, 0x8000, 0, 0x3F80],
                                       np.uint16)
    d["post"][1, :] = 2.0 ** -100
    want = orc.post(d["x"], d["residual"], d["post"], d["comb"])
    res = dev_bf16(d["residual"])
    ops.mhc_post(dev_bf16(d["x"]), res, dev_f32(d["post"]), dev_f32(d["comb"]), out=res)
    torch.cuda.synchronize()
    assert np.array_equal(host_bits(res), want)


# ------------------------------------------------------------------ boundary


# distinct per-group scales (pre, post, comb): a swapped group index on
# either side would show here
DISTINCT_SCALES = (0.25, 1.5, 3.0)


@pytest.mark.parametrize("scale", [(0.5, 0.5, 0.5), DISTINCT_SCALES])
def test_tiny_t4_h256_all_modes(scale):
    d = synth.workload_inputs("tiny_t4_h256", scale=scale)
    for mode in ("shifted", "unshifted", "pre"):
        g = run_gpu(mode, d)
        o = run_oracle(mode, d)
        compare(mode, g, o, d=d)


@pytest.mark.parametrize("T", synth.DECODE_TOKENS)
def test_decode_sweep_shifted_h7168(T):
    d = synth.make_inputs(**synth.decode_workload(T))
    g = run_gpu("shifted", d)
    o = run_oracle("shifted", d)
    compare("shifted", g, o, li_ulps=1)


@pytest.mark.parametrize("mode", ["shifted", "unshifted", "pre"])
@pytest.mark.parametrize("T", [1, 64])
def test_decode_distinct_scales_h7168(mode, T):
    """The single-wave forms, whose coefficients come from the 16-lane
    routine, with distinct per-group scales."""
    d = synth.make_inputs(**synth.decode_workload(T), scale=DISTINCT_SCALES)
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)


@pytest.mark.parametrize("mode", ["unshifted", "pre"])
@pytest.mark.parametrize("T", [1, 5, 32, 33, 64, 113, 128])
def test_decode_sweep_unshifted_h7168(mode, T):
    """Unshifted and pre-only calls of one tile at hidden 7168 (112 slices,
    at most 2 tokens per CTA): the streaming kernel forms the coefficients
    and its owner CTAs write the layer input. Up to 64 tokens the fused
    form's workers take the decode mapping (quarter units up to 32 tokens,
    whole units above). 113 tokens: one more than the slices, so a CTA has
    two tokens and others one."""
    d = synth.make_inputs(**synth.decode_workload(T))
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)


@pytest.mark.parametrize("mode", ["shifted", "unshifted", "pre"])
@pytest.mark.parametrize("T,H", [(129, 256), (200, 512), (333, 1024), (130, 4096)])
def test_ragged_tiles(mode, T, H):
    d = synth.make_inputs(T, H, seed=300 + T + H)
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)


@pytest.mark.parametrize("mode", ["shifted", "unshifted", "pre"])
@pytest.mark.parametrize("T", [256, 300, 1024])
def test_slice_plans_at_hidden_7168(mode, T):
    """Token counts whose plans differ at hidden 7168: 56 slices of 128 over
    two tiles, 32 slices of 224 over three tiles with a ragged tail (both a
    single wave), and 32 slices over eight tiles (two items per CTA). The
    shifted form forms the coefficients in the streaming kernel in every
    case; the others in a second kernel."""
    d = synth.make_inputs(T, 7168, seed=500 + T)
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)


@pytest.mark.parametrize("T,H", [(1301, 7168), (5000, 1024), (3001, 2048)])
def test_shifted_several_items_per_cta(T, H):
    """Shifted calls with several items per CTA, whose coefficients are formed
    by the streaming kernel's coefficient warps from 4-token groups: more
    than 28 slices (two copies per group) with a ragged last group, 8 slices
    (four groups per slice) and 16 slices with a ragged last group."""
    S, _ = ops.plan(T, H)
    assert (T + 127) // 128 * S > 152
    d = synth.make_inputs(T, H, seed=700 + T)
    g = run_gpu("shifted", d)
    o = run_oracle("shifted", d)
    compare("shifted", g, o, d=d)


@pytest.mark.parametrize("T", [385, 513])
def test_end_rounds_split_around_the_last_items(T):
    """Hidden 38912 plans 152 slices of 256, so a token group's records take
    over a third of the stage area and an end-of-call round holds two groups;
    CTAs 0-31 have one group per item and 4 (385 tokens) or 5 (513) items.
    The last two items' groups, copied once their tiles have published, then
    fill a later round on their own (4 items) or share one with an earlier
    item's group (5 items: a round straddles the two kinds)."""
    H = 38912
    S, _ = ops.plan(T, H)
    assert S == 152 and (T + 127) // 128 in (4, 5)
    d = synth.make_inputs(T, H, seed=760 + T)
    g = run_gpu("shifted", d)
    o = run_oracle("shifted", d)
    compare("shifted", g, o, d=d)


@pytest.mark.parametrize("scale", [(0.5, 0.5, 0.5), DISTINCT_SCALES])
@pytest.mark.parametrize("mode", ["pre", "unshifted", "shifted"])
def test_mid_batch_t512_h7168(mode, scale):
    d = synth.workload_inputs("mid_t512_h7168", scale=scale)
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)


@pytest.mark.parametrize("norm", ["bf16", None])
def test_norm_weight_variants(norm):
    d = synth.make_inputs(40, 512, seed=401)
    for mode in ("shifted", "unshifted", "pre"):
        g = run_gpu(mode, d, norm=norm)
        o = run_oracle(mode, d, norm=norm)
        compare(mode, g, o, d=d, norm=norm)


def test_in_place_residual():
    d = synth.make_inputs(70, 1024, seed=402)
    o = run_oracle("shifted", d)
    g = run_gpu("shifted", d, in_place=True)
    compare("shifted", g, o)


def test_zero_tokens_is_a_noop():
    w = ops.mhc_prepare_weight(torch.zeros(24, 4 * 256, device="cuda"))
    e = torch.empty(0, 4, 256, dtype=torch.bfloat16, device="cuda")
    ro, li, pr, po, cb = ops.mhc_boundary_fused(
        torch.empty(0, 256, dtype=torch.bfloat16, device="cuda"), e,
        torch.empty(0, 4, device="cuda"), torch.empty(0, 4, 4, device="cuda"), w,
        torch.ones(3, device="cuda"), torch.zeros(24, device="cuda"))
    torch.cuda.synchronize()
    assert ro.numel() == 0 and li.numel() == 0


def test_outputs_stay_inside_their_buffers():
    """Outputs written into the middle of guarded buffers: the guard bytes
    around them keep their canary pattern."""
    T, H = 131, 256
    d = synth.make_inputs(T, H, seed=403)
    G = 4096                                   # guard elements each side
    canary16 = 0x5A5A
    big_res = torch.full((G * 2 + T * 4 * H,), canary16, dtype=torch.int16, device="cuda")
    big_li = torch.full((G * 2 + T * H,), canary16, dtype=torch.int16, device="cuda")
    big_f = torch.full((3, G * 2 + T * 16), 12345.0, device="cuda")
    rout = big_res[G:G + T * 4 * H].view(torch.bfloat16).view(T, 4, H)
    li = big_li[G:G + T * H].view(torch.bfloat16).view(T, H)
    pre = big_f[0, G:G + T * 4].view(T, 4)
    post = big_f[1, G:G + T * 4].view(T, 4)
    comb = big_f[2, G:G + T * 16].view(T, 4, 4)
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    ops.mhc_boundary_fused(dev_bf16(d["x"]), dev_bf16(d["residual"]), dev_f32(d["post"]),
                           dev_f32(d["comb"]), w, dev_f32(d["scale"]), dev_f32(d["base"]),
                           dev_f32(d["norm_w"]), dev_f32(d["pre_lag"]), residual_out=rout,
                           layer_input=li, pre_out=pre, post_out=post, comb_out=comb)
    torch.cuda.synchronize()
    for big, n in ((big_res, T * 4 * H), (big_li, T * H)):
        assert torch.all(big[:G] == canary16) and torch.all(big[G + n:] == canary16)
    for i, n in enumerate((T * 4, T * 4, T * 16)):
        assert torch.all(big_f[i, :G] == 12345.0) and torch.all(big_f[i, G + n:] == 12345.0)
    o = run_oracle("shifted", d)
    assert np.array_equal(host_bits(rout), o["residual_out"])
    assert bf16_ulp_diff(host_bits(li), o["layer_input"]).max() <= 1


# ------------------------------------------------------------------ stress


@pytest.mark.parametrize("iters", [1, 5, 20])
def test_stress_t1024_h4096_sampled_and_deterministic(iters):
    d = synth.workload_inputs("stress_t1024_h4096")
    p = ops.Params(sinkhorn_iters=iters)
    rows = np.unique(np.concatenate([[0, 127, 128, 511, 1023],
                                     np.random.default_rng(iters).integers(0, 1024, 27)]))
    w = ops.mhc_prepare_weight(dev_f32(d["fn"]))
    runs = [run_gpu("shifted", d, params=p, weight=w) for _ in range(10)]
    ref = runs[0]
    for r in runs[1:]:
        assert torch.equal(r["residual_out_dev"], ref["residual_out_dev"])
        assert torch.equal(r["layer_input_dev"], ref["layer_input_dev"])
        for k in ("pre", "post", "comb"):
            assert np.array_equal(r[k].view(np.uint32), ref[k].view(np.uint32)), k
    o = run_oracle("shifted", d, params=p, rows=rows)
    compare("shifted", ref, o, rows=rows)
    # unshifted and pre-only on the same stress inputs
    for mode in ("unshifted", "pre"):
        g = run_gpu(mode, d, params=p, weight=w)
        o = run_oracle(mode, d, params=p, rows=rows)
        compare(mode, g, o, rows=rows, d=d, params=p)


# ------------------------------------------------------------------ full size


def test_prefill_t8192_h7168_sampled_tokens():
    """The benchmark's workload and launch configuration, checked on sampled
    tokens (first/last of tiles, the tail, random) against the oracle."""
    cfg = synth.WORKLOADS["prefill_t8192_h7168"]
    T, H = cfg["T"], cfg["H"]
    d = synth.make_inputs_device(T, H, cfg["seed"], "cuda")
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 4095, 4096, T - 2, T - 1],
                                     np.random.default_rng(8192).integers(0, T, 40)]))
    idx = torch.from_numpy(rows).cuda()
    d["residual"] = host_bits(d["residual_dev"][idx])
    d["x"] = host_bits(d["x_dev"][idx])
    g = run_gpu("shifted", d, dev_tensors={"residual": d["residual_dev"], "x": d["x_dev"]})
    sub = dict(d, post=d["post"][rows], comb=d["comb"][rows], pre_lag=d["pre_lag"][rows])
    o = run_oracle("shifted", sub)
    gsel = {k: (v[idx] if isinstance(v, torch.Tensor) else v) for k, v in g.items()
            if k not in ("partials",)}
    for k in ("pre", "post", "comb"):
        gsel[k] = g[k][rows]
    gsel["partials"] = g["partials"][:, rows]
    compare("shifted", gsel, o)


@pytest.mark.parametrize("mode", ["shifted", "unshifted", "pre"])
def test_large_token_count_sampled(mode):
    """32768 tokens x hidden 7168 (1.9 GB of residual, 7168 work items, 47 per
    CTA): offsets past 2^31 elements, checked on sampled tokens."""
    T, H = 32768, 7168
    d = synth.make_inputs_device(T, H, 9, "cuda")
    rows = np.unique(np.concatenate([[0, 127, 128, 16383, 16384, T - 129, T - 128, T - 1],
                                     np.random.default_rng(32768).integers(0, T, 24)]))
    idx = torch.from_numpy(rows).cuda()
    d["residual"] = host_bits(d["residual_dev"][idx])
    d["x"] = host_bits(d["x_dev"][idx])
    g = run_gpu(mode, d, dev_tensors={"residual": d["residual_dev"], "x": d["x_dev"]})
    sub = dict(d, post=d["post"][rows], comb=d["comb"][rows], pre_lag=d["pre_lag"][rows])
    o = run_oracle(mode, sub)
    gsel = {k: (v[idx] if isinstance(v, torch.Tensor) else v) for k, v in g.items()
            if k not in ("partials",)}
    for k in ("pre", "post", "comb"):
        gsel[k] = g[k][rows]
    gsel["partials"] = g["partials"][:, rows]
    compare(mode, gsel, o, d=sub)
    del d, g
    torch.cuda.empty_cache()


@pytest.mark.parametrize("mode", ["shifted", "unshifted", "pre"])
@pytest.mark.parametrize("T,H", [(1, 32), (130, 32), (3, 96), (77, 160), (129, 38912)])
def test_hidden_size_extremes(mode, T, H):
    """The smallest hidden (one 32-wide chunk: one slice, 128 tokens per
    item), odd chunk counts, and the largest hidden the shifted form plans
    with items of at most 8 chunks (152 slices of 256)."""
    d = synth.make_inputs(T, H, seed=900 + T + H)
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)


@pytest.mark.parametrize("mode", ["unshifted", "pre"])
def test_hidden_65536_items_of_sixteen_chunks(mode):
    """Hidden 65536 (the largest supported): 128 slices of 16 chunks, which
    only the unshifted forms plan (the shifted form's collapse buffer holds
    8 chunks and the call reports MHC_ERR_UNSUPPORTED)."""
    T, H = 5, 65536
    d = synth.make_inputs(T, H, seed=965)
    assert ops.plan(T, H) == (128, 512)
    g = run_gpu(mode, d)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)
    with pytest.raises(ops.MhcError) as e:
        run_gpu("shifted", d)
    assert e.value.code == 4


# ------------------------------------------------------------------ stream capture


@pytest.mark.parametrize("T,H", [(64, 7168), (2048, 7168)])
def test_calls_capture_into_a_cuda_graph_and_replay_with_new_inputs(T, H):
    """The entry points allocate nothing and never synchronise, so a decode
    loop can capture them into a CUDA graph. Replaying the graph after new
    inputs were written into the same buffers gives the eager results for
    those inputs bit for bit (a single-wave and a multi-item plan; shifted,
    unshifted and pre-only forms), so no per-call state is frozen into the
    graph."""
    dev = "cuda"
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    A = synth.make_inputs(T, H, seed=610 + T)
    B = synth.make_inputs(T, H, seed=611 + T)
    keys_bf, keys_f = ("residual", "x"), ("post", "comb", "pre_lag")
    inp = {k: bf(A[k]) for k in keys_bf} | {k: f32(A[k]) for k in keys_f}
    scale, base, nw = f32(A["scale"]), f32(A["base"]), f32(A["norm_w"])
    w = ops.mhc_prepare_weight(f32(A["fn"]))
    ws = torch.empty(ops.workspace_bytes(T, H), dtype=torch.uint8, device=dev)

    def new_outs():
        o = {}
        for form in ("s", "u", "p"):
            o[form] = dict(layer_input=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                           pre_out=torch.empty(T, 4, device=dev),
                           post_out=torch.empty(T, 4, device=dev),
                           comb_out=torch.empty(T, 4, 4, device=dev))
            if form != "p":
                o[form]["residual_out"] = torch.empty_like(inp["residual"])
        return o

    def run(o, stream=None):
        for form, pl in (("s", inp["pre_lag"]), ("u", None)):
            ops.mhc_boundary_fused(inp["x"], inp["residual"], inp["post"], inp["comb"], w, scale,
                                   base, nw, pl, workspace=ws, stream=stream, **o[form])
        ops.mhc_pre(inp["residual"], w, scale, base, nw, workspace=ws, stream=stream, **o["p"])

    def load(d):
        for k in keys_bf:
            inp[k].copy_(bf(d[k]))
        for k in keys_f:
            inp[k].copy_(f32(d[k]))

    load(B)
    eager = new_outs()
    run(eager)
    torch.cuda.synchronize()
    load(A)
    cap = new_outs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(cap, stream=s)                       # warm-up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            run(cap, stream=s)
    torch.cuda.synchronize()
    g.replay()                                   # inputs A
    torch.cuda.synchronize()
    load(B)
    for o in cap.values():
        for v in o.values():
            v.zero_()
    torch.cuda.synchronize()
    g.replay()                                   # inputs B, same buffers
    torch.cuda.synchronize()
    assert ops.mhc_get_device_status() == 0
    for form in cap:
        for k, v in eager[form].items():
            got = cap[form][k]
            if v.dtype == torch.bfloat16:
                v, got = v.view(torch.int16), got.view(torch.int16)
            assert torch.equal(v, got), (form, k)


@pytest.mark.parametrize("T,H", [(64, 7168), (512, 7168), (2048, 7168)])
def test_captured_chain_of_shifted_calls_sharing_a_workspace(T, H):
    """Three shifted calls captured back to back into one graph share one
    workspace, each reading the residual the one before it wrote. Each call
    needs a flag value of its own: one that took the previous call's would
    find every flag already set and read that call's partials, formed from
    another residual. Replayed twice, the chain gives the eager chain's
    results bit for bit. Plans: one tile, several tiles in a single wave,
    several items per CTA."""
    dev = "cuda"
    n = 3
    bf = lambda a: torch.from_numpy(np.ascontiguousarray(a)).view(torch.bfloat16).to(dev)
    f32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.float32)).to(dev)
    A = synth.make_inputs(T, H, seed=720 + T)
    res0, x = bf(A["residual"]), bf(A["x"])
    post, comb, pl = f32(A["post"]), f32(A["comb"]), f32(A["pre_lag"])
    scale, base, nw = f32(A["scale"]), f32(A["base"]), f32(A["norm_w"])
    w = ops.mhc_prepare_weight(f32(A["fn"]))
    ws = torch.empty(ops.workspace_bytes(T, H), dtype=torch.uint8, device=dev)

    def new_outs():
        return [dict(residual_out=torch.empty_like(res0),
                     layer_input=torch.empty(T, H, dtype=torch.bfloat16, device=dev),
                     pre_out=torch.empty(T, 4, device=dev), post_out=torch.empty(T, 4, device=dev),
                     comb_out=torch.empty(T, 4, 4, device=dev)) for _ in range(n)]

    def chain(outs, stream=None):
        r = res0
        for o in outs:
            ops.mhc_boundary_fused(x, r, post, comb, w, scale, base, nw, pl, workspace=ws,
                                   stream=stream, **o)
            r = o["residual_out"]

    eager = new_outs()
    chain(eager)
    torch.cuda.synchronize()
    cap = new_outs()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain(cap, stream=s)                     # warm-up on the capture stream
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            chain(cap, stream=s)
    torch.cuda.synchronize()
    for _ in range(2):
        for o in cap:
            for v in o.values():
                v.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert ops.mhc_get_device_status() == 0
        for k in range(n):
            for key, v in eager[k].items():
                got = cap[k][key]
                if v.dtype == torch.bfloat16:
                    v, got = v.view(torch.int16), got.view(torch.int16)
                assert torch.equal(v, got), (k, key)


# ------------------------------------------------------------------ reciprocal


def test_coefficient_reciprocal_is_correctly_rounded_for_every_normal_input():
    """The coefficients divide through the "mhc_boundary" page's rcp (hardware
    approximation plus one Newton-Raphson step), the oracle through an IEEE
    division. Exhaustively, for every positive normal x whose reciprocal is
    normal (2^-126 <= x <= 2^126: sums of Sinkhorn rows and columns, softmax
    sums, sigmoid denominators clamped at 2^126), the two are the same
    float."""
    lo, hi = 0x00800000, 0x7E800000
    n, first = ops.mhc_debug_rcp_check(lo, hi - lo + 1)
    assert n == 0, f"{n} patterns differ, first {first:#010x}"


# ------------------------------------------------------------------ bounded waits


def test_unarmed_wait_times_out_and_context_survives():
    ops.mhc_set_wait_timeout_ns(20_000_000)          # 20 ms
    try:
        ops.mhc_debug_unarmed_wait()
        assert ops.mhc_get_device_status() == 7
        assert ops.mhc_last_timeout_site() == 99
        assert ops.mhc_get_device_status() == 0       # read clears the word
    finally:
        ops.mhc_set_wait_timeout_ns(0)
    d = synth.make_inputs(4, 256, seed=404)
    compare("shifted", run_gpu("shifted", d), run_oracle("shifted", d))


@pytest.mark.parametrize("mode,T,H,in_place", [("unshifted", 5, 7168, True), ("unshifted", 3, 16384, False),
                                               ("pre", 3, 16384, False), ("unshifted", 40, 8192, False),
                                               ("pre", 128, 8192, False)])
def test_unshifted_single_wave_collapse_paths(mode, T, H, in_place):
    """Unshifted single-wave calls write the layer input in the streaming
    kernel up to hidden 8192 (the owner CTA recomputes each token's updated
    residual); in place, or above hidden 8192, the collapse kernel still
    follows. Both against the oracle."""
    d = synth.make_inputs(T, H, seed=2100 + T + H)
    g = run_gpu(mode, d, in_place=in_place)
    o = run_oracle(mode, d)
    compare(mode, g, o, d=d)
