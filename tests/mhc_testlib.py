"""Helpers shared by the GPU parity tests: moving the seeded inputs to the
device, running the library through its C ABI, and comparing with the CPU
oracle at the tolerances stated in the tests."""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
from manifold_constrained_hyper_gb300 import ops

MODES = {"pre": orc.MODE_PRE_ONLY, "unshifted": orc.MODE_FUSED_UNSHIFTED,
         "shifted": orc.MODE_FUSED_SHIFTED}

# Tolerances. Coefficients: 1e-5 relative (the fp32 arithmetic of sigmoid,
# softmax and a 20-step Sinkhorn on both sides, with libm's and CUDA's exp,
# leaves a few fp32 ulps), plus 1e-7 absolute for values near zero. Mixes:
# 1e-5 of the larger of |mix| and the 2-norm of its 4H terms (a mix near zero
# is a sum that cancelled, whose error scales with its terms, not itself).
COEF_RTOL, COEF_ATOL = 1e-5, 1e-7      # pre, post, comb
MIX_RTOL = 1e-5                         # |g - o| <= 1e-5 * max(|o|, ||terms||_2)


def dev_bf16(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)


def dev_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between bit patterns (+0 and -0 coincide)."""
    def ordered(u):
        v = u.astype(np.int32)
        return np.where(v & 0x8000, -(v & 0x7FFF), v)
    return np.abs(ordered(a) - ordered(b))


def run_gpu(mode: str, d: dict, norm: str = "f32", params: ops.Params | None = None,
            weight=None, in_place: bool = False, dev_tensors: dict | None = None):
    """Runs one boundary call on the GPU. `d` holds numpy inputs (synth);
    `dev_tensors` may carry residual/x already on the device. Returns a dict
    of numpy outputs plus the workspace partials as [S][T][25]."""
    dev_tensors = dev_tensors or {}
    res = dev_tensors.get("residual")
    if res is None:
        res = dev_bf16(d["residual"])
    T, _, H = res.shape
    fn = dev_f32(d["fn"])
    w = weight if weight is not None else ops.mhc_prepare_weight(fn)
    scale, base = dev_f32(d["scale"]), dev_f32(d["base"])
    nw = None
    if norm == "f32":
        nw = dev_f32(d["norm_w"])
    elif norm == "bf16":
        nw = dev_bf16(orc.f32_to_bf16(d["norm_w"]))
    ws = torch.empty(max(ops.workspace_bytes(T, H), 16), dtype=torch.uint8, device="cuda")
    out = {}
    if mode == "pre":
        li, pr, po, cb = ops.mhc_pre(res, w, scale, base, nw, params, workspace=ws)
    else:
        x = dev_tensors.get("x")
        if x is None:
            x = dev_bf16(d["x"])
        pl = dev_f32(d["pre_lag"]) if mode == "shifted" else None
        rout = res if in_place else None
        ro, li, pr, po, cb = ops.mhc_boundary_fused(
            x, res, dev_f32(d["post"]), dev_f32(d["comb"]), w, scale, base, nw, pl, params,
            residual_out=rout, workspace=ws)
        out["residual_out_dev"] = ro
    torch.cuda.synchronize()
    assert ops.mhc_get_device_status() == 0
    if mode == "shifted" and not (params and params.batch_invariant) and ops.plan_cluster(T, H):
        # a cluster call keeps each token's reduced values (24 mixes, the 4H
        # sum of squares, padding) at bytes 256 .. 256 + 112 T: one "slice"
        part = ws[256: 256 + T * 112].view(torch.float32).view(1, T, 28)[..., :25]
        out.update(layer_input_dev=li, pre=pr.cpu().numpy(), post=po.cpu().numpy(),
                   comb=cb.cpu().numpy(), partials=part.cpu().numpy(), path="cluster")
        return out
    S, _ = ops.plan(T, H)
    # the library's internal partials, 25 values per token and slice (24
    # mixes, then the 4H sum of squares), in a block of 128 x 32 floats per
    # (128-token tile, slice) item: token-major [128][28] when the streaming
    # kernel's workers reduce them (a single wave of items; for the unshifted
    # forms only one tile whose CTAs have at most 5 tokens each, one round);
    # value-major [25][128] in the other unshifted calls; otherwise (shifted,
    # several items per CTA) one 32-float record per token and slice,
    # [tiles * 128][S][32]
    tiles = (T + 127) // 128
    sms = min(152, torch.cuda.get_device_properties(0).multi_processor_count)
    # (the partials start 256 bytes into the workspace, after the epoch cell)
    raw = ws[256: 256 + tiles * S * 32 * 128 * 4].view(torch.float32).view(tiles, S, 32 * 128)
    single_wave = tiles * S <= sms and not (params and params.batch_invariant)
    in_kernel = single_wave and (mode == "shifted" or (tiles == 1 and -(-T // S) <= 5))
    if in_kernel:
        blk = raw[..., : 128 * 28].reshape(tiles, S, 128, 28)[..., :25].permute(1, 0, 2, 3)
    elif mode == "shifted":
        blk = raw.reshape(tiles * 128, S, 32)[..., :25].permute(1, 0, 2)
    else:
        blk = raw[..., : 25 * 128].reshape(tiles, S, 25, 128).permute(1, 0, 3, 2)
    part = blk.reshape(S, tiles * 128, 25)[:, :T, :].cpu().numpy()
    out.update(layer_input_dev=li, pre=pr.cpu().numpy(), post=po.cpu().numpy(),
               comb=cb.cpu().numpy(), partials=part, path="slices")
    return out


def gpu_mixes(partials: np.ndarray) -> np.ndarray:
    """Sum of the slice partials in slice order, in fp32 (as the finishing
    kernel does): [T, 24]."""
    acc = np.zeros(partials.shape[1:], np.float32)
    for s in range(partials.shape[0]):
        acc = (acc + partials[s]).astype(np.float32)
    return acc[:, :24]


def run_oracle(mode: str, d: dict, norm: str = "f32", params: ops.Params | None = None,
               rows=None):
    p = params or ops.Params()
    op = orc.OracleParams(p.hc_norm_eps, p.hc_pre_eps, p.hc_post_mult, p.sinkhorn_eps,
                          p.norm_eps, p.sinkhorn_iters)
    nw = None
    if norm == "f32":
        nw = d["norm_w"]
    elif norm == "bf16":
        nw = orc.f32_to_bf16(d["norm_w"])
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    kw = {}
    if mode != "pre":
        kw = dict(x=sel(d["x"]), post_mix=sel(d["post"]), comb=sel(d["comb"]))
        if mode == "shifted":
            kw["pre_lag"] = sel(d["pre_lag"])
    return orc.boundary(MODES[mode], sel(d["residual"]), d["fn"], d["scale"], d["base"], nw,
                        params=op, **kw)


def oracle_layer_input_given_pre(mode: str, d: dict, pre: np.ndarray, norm="f32",
                                 params=None, rows=None):
    """The oracle's layer input when the collapse uses the given `pre` [T, 4]
    (the GPU's own, for the unshifted forms): the unshifted boundary equals
    the shifted one fed its own pre, and pre-only equals the shifted one with
    an identity update (x = 0, post = 0, comb = I; a bitwise copy of normal
    bf16 values)."""
    dd = dict(d)
    dd["pre_lag"] = np.ascontiguousarray(pre, np.float32)
    if mode == "pre":
        T = d["residual"].shape[0]
        dd["x"] = np.zeros(d["residual"].shape[::2], np.uint16)
        dd["post"] = np.zeros((T, 4), np.float32)
        dd["comb"] = np.broadcast_to(np.eye(4, dtype=np.float32), (T, 4, 4)).copy()
    return run_oracle("shifted", dd, norm, params, rows)["layer_input"]


def _f64(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def _ulp(v: np.ndarray) -> np.ndarray:
    """One bf16 ulp at the magnitude of v (8 significant bits)."""
    return np.ldexp(1.0, np.frexp(np.maximum(np.abs(v), 2.0 ** -126))[1] - 8)


def _unshifted_li_excess(mode, d, g, o, li_gpu, norm, rows):
    """Largest ratio of |out_gpu - out_oracle| to the element's derived bound
    (see compare): <= 1 means every element is within its bound."""
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    stream = host_bits(g["residual_out_dev"]) if mode == "unshifted" else sel(d["residual"])
    if mode == "unshifted":
        stream = sel(stream)
    r = _f64(stream)                                             # [t, 4, H]
    p_o = o["pre"].astype(np.float64)
    p_g = sel(g["pre"]).astype(np.float64)
    # the two exact collapse sums are at most E apart; each side forms its
    # own as a 4-step fp32 FMA chain (4 roundings, each at most 2^-24 of the
    # chain's largest partial, itself at most sum_j |p_j r_j|)
    mag = np.einsum("tj,tjh->th", np.abs(p_o), np.abs(r))
    E = np.einsum("tj,tjh->th", np.abs(p_g - p_o), np.abs(r)) + 8 * 2.0 ** -24 * mag
    li_o = np.einsum("tj,tjh->th", p_o, r)
    if norm is None:
        scale = np.ones_like(li_o)
    else:
        w = d["norm_w"].astype(np.float64)
        if norm == "bf16":
            w = _f64(orc.f32_to_bf16(d["norm_w"]))
        scale = o["rstd_li"].astype(np.float64)[:, None] * np.abs(w)[None, :]
    out_o = _f64(o["layer_input"])
    bound = 2 * _ulp(out_o) + (E + _ulp(np.abs(li_o) + E)) * scale
    err = np.abs(_f64(li_gpu) - out_o)
    return float(np.max(err / bound)) if err.size else 0.0


def compare(mode: str, g: dict, o: dict, rows=None, li_ulps: int = 1, mixes: bool = True,
            d: dict | None = None, norm="f32", params=None):
    """Element-wise comparison of GPU outputs (optionally the token `rows`)
    with the oracle's. Returns a dict of observed error figures.

    Layer input: shifted, the collapse is exact on both sides and the bar is
    1 bf16 ulp against the oracle. Unshifted / pre-only, the collapse uses
    this boundary's pre, which the two sides form in different summation
    orders (checked separately at 1e-5); where sum_j pre_j r_j cancels, that
    difference is amplified in ulps. So the bar there is: 1 ulp against the
    oracle's layer input computed from the GPU's own pre; at least 99.9 % of
    elements within 1 ulp of the independent oracle; and every element
    within a bound derived from the pre difference: with
    E = sum_j |pre_gpu_j - pre_oracle_j| |r_j| + 8 * 2^-24 * sum_j |pre_j r_j|
    (how far the two collapse sums can be apart: the pre difference, and
    each side's 4-step fp32 FMA chain), |out_gpu - out_oracle| <=
    2 ulp(out) + (E + ulp(|li| + E)) * rstd_li * |norm_w|, li = sum_j pre_j r_j
    (the roundings of li and of the output on each side, and the sums'
    spread carried through the normalisation). The count of elements
    beyond 1 ulp and the largest distance are recorded in the stats."""
    sel = (lambda a: a) if rows is None else (lambda a: a[rows])
    stats = {}
    if mode != "pre":
        ro = sel(host_bits(g["residual_out_dev"]))
        assert np.array_equal(ro, o["residual_out"]), "residual_out differs"
    li = sel(host_bits(g["layer_input_dev"]))
    du = bf16_ulp_diff(li, o["layer_input"])
    stats["li_max_ulp"] = int(du.max()) if du.size else 0
    stats["li_frac_exact"] = float(np.mean(du == 0)) if du.size else 1.0
    stats["li_n_beyond_1ulp"] = int(np.sum(du > 1))
    if mode == "shifted":
        assert stats["li_max_ulp"] <= li_ulps, stats
    else:
        assert d is not None, "unshifted comparison needs the inputs"
        assert float(np.mean(du <= 1)) >= 0.999, stats
        ref = oracle_layer_input_given_pre(mode, d, g["pre"], norm, params, rows)
        dc = bf16_ulp_diff(li, ref)
        stats["li_max_ulp_given_pre"] = int(dc.max()) if dc.size else 0
        assert stats["li_max_ulp_given_pre"] <= 1, stats
        over = _unshifted_li_excess(mode, d, g, o, li, norm, rows)
        stats["li_max_over_bound"] = over
        assert over <= 1.0, stats
    for k in ("pre", "post", "comb"):
        gv, ov = sel(g[k]).astype(np.float64), o[k].astype(np.float64)
        err = np.abs(gv - ov)
        bound = COEF_RTOL * np.abs(ov) + COEF_ATOL
        stats[k + "_max_rel"] = float(np.max(err / np.maximum(np.abs(ov), 1e-30)))
        assert np.all(err <= bound), (k, float(np.max(err - bound)))
    if mixes:
        gm = sel(gpu_mixes(g["partials"])).astype(np.float64)
        om = o["mix"].astype(np.float64)
        scale = np.maximum(np.abs(om), o["mix_scale"].astype(np.float64))
        err = np.abs(gm - om)
        stats["mix_max_scaled"] = float(np.max(err / scale))
        assert np.all(err <= MIX_RTOL * scale), stats["mix_max_scaled"]
    return stats
