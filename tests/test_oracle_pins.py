"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Sources of truth used here (none re-types the oracle's formulas):
* torch's fp32 -> bf16 conversion (round to nearest even) as a library routine;
* exact rational arithmetic (``fractions.Fraction``) for the mixer contraction;
* arithmetic (not bit-level) rounding for TF32;
* closed forms of special cases (identity comb, one-hot mixer, constant
  rows, uniform logits, zero mixer, saturation);
* invariants the pages state (hi + lo == TF32 exactly, comb non-negative
  with columns summing to S/(S + eps) after the last column step, pre in
  (eps, 1 + eps], post in (0, 2]).
Page references: "mhc_boundary" is the vLLM DeepSeek-V4.1 shifted mHC
boundary API page, "pre study" is "The Hyper Connection Preprocessing GPU
Kernel Study".
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle as orc
from manifold_constrained_hyper_gb300 import synth

B2F = synth.bf16_bits_to_float


def torch_bf16(a):
    """Library routine: torch's RNE fp32 -> bf16 conversion, as bits."""
    t = torch.from_numpy(np.ascontiguousarray(a, np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32(u):
    return np.array([u], np.uint32).view(np.float32)[0]


def bits(f):
    return int(np.array([f], np.float32).view(np.uint32)[0])


# ---------------------------------------------------------------- bf16 / ftz


def test_bf16_rne_hand_cases():
    cases = {
        1.0: 0x3F80,
        1.0 + 2.0 ** -8: 0x3F80,                  # tie -> even (down)
        1.0 + 3 * 2.0 ** -8: 0x3F82,              # tie -> even (up)
        1.0 + 2.0 ** -8 + 2.0 ** -20: 0x3F81,     # above the tie
        -(1.0 + 2.0 ** -8): 0xBF80,
        f32(0x00018000): 0x0002,                  # subnormal tie, odd -> up
        f32(0x00008000): 0x0000,                  # subnormal tie, even -> down
        f32(0x7F7FFFFF): 0x7F80,                  # overflows to +inf
    }
    got = orc.f32_to_bf16(np.array(list(cases.keys()), np.float32))
    assert [int(v) for v in got] == list(cases.values())


def test_bf16_matches_torch_on_random_bits():
    rng = np.random.default_rng(7)
    u = rng.integers(0, 2 ** 32, size=200_000, dtype=np.uint64).astype(np.uint32)
    f = u.view(np.float32)
    f = f[np.isfinite(f)]
    assert np.array_equal(orc.f32_to_bf16(f), torch_bf16(f))


# ---------------------------------------------------------------- TF32 split


def tf32_arith(w):
    """Round to 10 explicit mantissa bits, ties away from zero, by arithmetic."""
    if w == 0.0:
        return w
    m, e = math.frexp(abs(w))            # |w| = m * 2^e, m in [0.5, 1)
    q = abs(w) / 2.0 ** (e - 11)         # 11 significant bits above the point
    r = math.floor(q + 0.5) * 2.0 ** (e - 11)
    return math.copysign(r, w)


def test_tf32_round_hand_cases():
    cases = [
        (0x3F801000, 0x3F802000),   # 1 + 2^-11: exact tie, away from zero
        (0xBF801000, 0xBF802000),   # negative tie, away from zero
        (0x3F800FFF, 0x3F800000),   # just below the tie
        (0x3FFFF000, 0x40000000),   # carry into the exponent
        (0x3F801FFF, 0x3F802000),
    ]
    w = np.array([c[0] for c in cases], np.uint32).view(np.float32)
    got = orc.tf32_round(w).view(np.uint32)
    assert [int(v) for v in got] == [c[1] for c in cases]


def test_tf32_round_matches_arithmetic_rounding():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal(20_000) * np.exp(rng.uniform(-30, 30, 20_000))).astype(np.float32)
    got = orc.tf32_round(w)
    want = np.array([tf32_arith(float(v)) for v in w], np.float32)
    assert np.array_equal(got, want)


def test_hi_lo_split_is_exact():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal(100_000) / 64).astype(np.float32)
    r, hi, lo = orc.tf32_split(w)
    hif, lof = B2F(hi).astype(np.float64), B2F(lo).astype(np.float64)
    assert np.array_equal(hif + lof, r.astype(np.float64))          # exact
    assert np.array_equal(hi, torch_bf16(r))                          # hi = bf16(r)
    # lo is at most half an ulp of hi (8 significant bits)
    ulp_hi = np.exp2(np.floor(np.log2(np.abs(hif))) - 7)
    assert np.all(np.abs(lof) <= ulp_hi / 2)


def test_weight_tiles_unswizzle_reconstructs_hi_lo():
    H = 64
    rng = np.random.default_rng(5)
    fn = (rng.standard_normal((24, 4 * H)) / 16).astype(np.float32)
    tiles = orc.weight_tiles(fn, H)
    _, hi, lo = orc.tf32_split(fn)
    stacked = np.concatenate([hi, lo], axis=0)            # [48, 4H]
    t = tiles.reshape(H // 32, 4, 48, 4, 8)                # chunk, stream, row, unit, elem
    rows = np.arange(48)
    back = np.empty_like(t)
    for p in range(4):                                     # physical unit p holds
        logical = p ^ ((rows >> 1) & 3)                    # logical unit p ^ swz(row)
        back[:, :, rows, logical, :] = t[:, :, rows, p, :]
    # back[c, s, r, u, i] = stacked[r, s*H + 32c + 8u + i]
    want = stacked.reshape(48, 4, H // 32, 4, 8).transpose(2, 1, 0, 3, 4)
    assert np.array_equal(back, want)


# ---------------------------------------------------------------- residual update


def _bf16(a):
    return torch_bf16(np.asarray(a, np.float32))


def test_update_identity_comb_zero_post_is_copy():
    d = synth.make_inputs(3, 64, seed=21)
    comb = np.broadcast_to(np.eye(4, dtype=np.float32), (3, 4, 4))
    out = orc.post(d["x"], d["residual"], np.zeros((3, 4), np.float32), comb)
    assert np.array_equal(out, d["residual"])


def test_update_identity_comb_unit_post_zero_residual_is_x():
    d = synth.make_inputs(3, 64, seed=22)
    comb = np.broadcast_to(np.eye(4, dtype=np.float32), (3, 4, 4))
    out = orc.post(d["x"], np.zeros_like(d["residual"]), np.ones((3, 4), np.float32), comb)
    for s in range(4):
        assert np.array_equal(out[:, s], d["x"])


def test_update_comb_orientation():
    # comb[j][s] multiplies residual stream j into stream s: one off-diagonal
    # 1 at j=0, s=1 sends stream 0 into stream 1 and nothing else anywhere.
    d = synth.make_inputs(2, 64, seed=23)
    comb = np.zeros((2, 4, 4), np.float32)
    comb[:, 0, 1] = 1.0
    out = orc.post(d["x"], d["residual"], np.zeros((2, 4), np.float32), comb)
    assert np.array_equal(out[:, 1], d["residual"][:, 0])
    for s in (0, 2, 3):
        assert not np.any(out[:, s] & 0x7FFF)


def test_update_within_one_ulp_of_exact():
    d = synth.make_inputs(4, 256, seed=24)
    out = orc.post(d["x"], d["residual"], d["post"], d["comb"])
    r = B2F(d["residual"]).astype(np.float64)
    x = B2F(d["x"]).astype(np.float64)
    exact = (d["post"][:, :, None] * x[:, None, :]
             + np.einsum("tjs,tjh->tsh", d["comb"].astype(np.float64), r))
    want = _bf16(exact.astype(np.float32))
    diff = np.abs(out.astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1 and np.mean(diff == 0) > 0.99


def test_update_flushes_subnormals():
    T, H = 1, 32
    x = np.zeros((T, H), np.uint16)
    res = np.zeros((T, 4, H), np.uint16)
    x[0, 0] = bits(2.0 ** -30) >> 16                   # post*x = 2^-130: subnormal
    res[0, 0, 1] = 0x0001                              # a subnormal bf16 input
    res[0, 0, 2] = bits(2.0 ** -120) >> 16             # comb*res = 2^-128: subnormal
    post = np.full((T, 4), 2.0 ** -100, np.float32)
    comb = np.zeros((T, 4, 4), np.float32)
    comb[0, 0, 0] = 1.0
    comb[0, 0, 1] = 2.0 ** -8
    out = orc.post(x, res, post, comb)
    assert out[0, 0, 0] == 0 and out[0, 0, 1] == 0 and out[0, 1, 2] == 0
    # a normal result is kept
    x[0, 3] = bits(1.0) >> 16
    post[:] = 1.0
    out = orc.post(x, res, post, comb)
    assert out[0, 0, 3] == 0x3F80


# ---------------------------------------------------------------- mixer, rstd


def _pre_only(res, fn, base=None, norm_w=None, params=None):
    H = res.shape[2]
    base = np.zeros(24, np.float32) if base is None else base
    return orc.boundary(orc.MODE_PRE_ONLY, res, fn, np.array([0.5] * 3, np.float32),
                        base, norm_w, params=params)


def test_mixer_matches_exact_rational_sum():
    T, H = 2, 32
    d = synth.make_inputs(T, H, seed=31)
    out = _pre_only(d["residual"], d["fn"])
    r = orc.tf32_round(d["fn"])
    cur = B2F(d["residual"]).reshape(T, 4 * H)
    for t in range(T):
        for n in range(24):
            exact = sum(Fraction(float(a)) * Fraction(float(b))
                        for a, b in zip(r[n], cur[t]))
            want = np.float32(float(exact))
            got = out["mix"][t, n]
            assert abs(float(got) - float(exact)) <= abs(float(want)) * 2.0 ** -23 + 1e-30


def test_mixer_zero_weight_gives_zero():
    d = synth.make_inputs(2, 64, seed=32)
    out = _pre_only(d["residual"], np.zeros((24, 256), np.float32))
    assert np.all(out["mix"] == 0.0)


def test_mixer_one_hot_picks_flattened_column():
    # fn[n][s*H + h] selects stream s, hidden h of the token
    T, H = 2, 64
    d = synth.make_inputs(T, H, seed=33)
    w = np.float32(1.0 + 2.0 ** -11 + 2.0 ** -20)      # rounds (away) in TF32
    for n, s, h in [(0, 0, 5), (7, 1, 17), (13, 2, 63), (23, 3, 0)]:
        fn = np.zeros((24, 4 * H), np.float32)
        fn[n, s * H + h] = w
        out = _pre_only(d["residual"], fn)
        want = orc.tf32_round(np.array([w]))[0] * B2F(d["residual"][:, s, h])
        assert np.array_equal(out["mix"][:, n], want.astype(np.float32))
        others = np.delete(out["mix"], n, axis=1)
        assert np.all(others == 0.0)


def test_rstd_of_constant_rows():
    T, H = 3, 64
    c = np.array([0.5, 3.0, 1.0 / 128], np.float32)
    res = np.broadcast_to(_bf16(c)[:, None, None], (T, 4, H)).copy()
    out = _pre_only(res, np.zeros((24, 4 * H), np.float32))
    cf = B2F(_bf16(c)).astype(np.float64)
    want = 1.0 / np.sqrt(cf * cf + 1e-6)
    assert np.allclose(out["rstd"], want, rtol=2e-7, atol=0)


# ---------------------------------------------------------------- coefficients


def sigmoid64(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


def test_zero_mixer_coefficients_closed_form():
    T, H = 2, 64
    d = synth.make_inputs(T, H, seed=41, base_std=1.0)
    out = _pre_only(d["residual"], np.zeros((24, 4 * H), np.float32), base=d["base"])
    b = d["base"].astype(np.float64)
    assert np.allclose(out["pre"], sigmoid64(b[:4]) + 1e-6, rtol=3e-7, atol=0)
    assert np.allclose(out["post"], 2.0 * sigmoid64(b[4:8]), rtol=3e-7, atol=0)


def test_uniform_logits_give_uniform_comb():
    # equal logits: softmax gives 1/4 + eps everywhere, and every Sinkhorn
    # step maps an all-equal matrix v to v / (4v + eps)
    T, H = 1, 32
    res = np.zeros((T, 4, H), np.uint16)
    base = np.zeros(24, np.float32)
    base[8:] = 0.7
    for iters in (1, 2, 5, 20):
        out = _pre_only(res, np.zeros((24, 4 * H), np.float32), base=base,
                        params=orc.OracleParams(sinkhorn_iters=iters))
        v = 0.25 + 1e-6
        for _ in range(2 * iters - 1):
            v = v / (4 * v + 1e-6)
        assert np.allclose(out["comb"], v, rtol=1e-6, atol=0)


def test_sigmoid_saturation_and_clamp():
    got = orc.sigmoid(np.array([0.0, 20.0, -100.0, -200.0, 3.0], np.float32))
    assert got[0] == 0.5
    assert got[1] == 1.0                                  # saturates in fp32
    assert got[2] == np.float32(2.0 ** -126)               # clamped denominator
    assert got[3] == np.float32(2.0 ** -126)
    assert abs(got[4] - sigmoid64(3.0)) <= 2 ** -23


def test_coefficient_invariants_and_sinkhorn_convergence():
    d = synth.make_inputs(64, 256, seed=42, base_std=1.0)
    out = orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"], d["fn"], d["scale"],
                       d["base"], d["norm_w"], x=d["x"], post_mix=d["post"],
                       comb=d["comb"], pre_lag=d["pre_lag"])
    eps = 1e-6
    assert np.all(out["pre"] > eps) and np.all(out["pre"] <= 1 + eps)
    assert np.all(out["post"] > 0) and np.all(out["post"] <= 2)
    c = out["comb"].astype(np.float64)
    assert np.all(c >= 0)
    cols = c.sum(axis=1)                                  # sum over rows i
    assert np.allclose(cols, 1.0, atol=4e-6)              # S/(S+eps) ~ 1 - eps
    rows = c.sum(axis=2)
    assert np.allclose(rows, 1.0, atol=1e-3)              # converged after 20


def test_sinkhorn_single_iteration_normalises_columns_only():
    rng = np.random.default_rng(43)
    c = rng.uniform(0.05, 1.0, (32, 16)).astype(np.float32)
    out = orc.sinkhorn(c, 1, 1e-6).reshape(32, 4, 4).astype(np.float64)
    s = c.reshape(32, 4, 4).astype(np.float64).sum(axis=1)
    assert np.allclose(out.sum(axis=1), s / (s + 1e-6), rtol=1e-6)
    # rows are the inputs scaled per column, not renormalised
    assert np.allclose(out, c.reshape(32, 4, 4) / (s + 1e-6)[:, None, :], rtol=1e-6)


def test_stream_permutation_equivariance():
    T, H = 3, 64
    d = synth.make_inputs(T, H, seed=44)
    perm = np.array([2, 0, 3, 1])
    kp = (perm[:, None] * H + np.arange(H)[None, :]).reshape(-1)
    rows = np.concatenate([perm, 4 + perm, 8 + (4 * perm[:, None] + perm[None, :]).reshape(-1)])
    args = dict(params=orc.OracleParams())
    a = orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"], d["fn"], d["scale"], d["base"],
                     d["norm_w"], x=d["x"], post_mix=d["post"], comb=d["comb"],
                     pre_lag=d["pre_lag"], **args)
    b = orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"][:, perm], d["fn"][rows][:, kp],
                     d["scale"], d["base"][rows], d["norm_w"], x=d["x"],
                     post_mix=d["post"][:, perm], comb=d["comb"][:, perm][:, :, perm],
                     pre_lag=d["pre_lag"][:, perm], **args)
    assert np.array_equal(b["residual_out"], a["residual_out"][:, perm])
    assert np.allclose(b["mix"], a["mix"][:, rows], rtol=1e-6, atol=1e-7)
    assert np.allclose(b["pre"], a["pre"][:, perm], rtol=1e-5)
    assert np.allclose(b["post"], a["post"][:, perm], rtol=1e-5)
    assert np.allclose(b["comb"], a["comb"][:, perm][:, :, perm], rtol=1e-5, atol=1e-7)


# ---------------------------------------------------------------- collapse + RMSNorm


def _shifted(d, pre_lag, norm_w=None, comb=None, post=None):
    return orc.boundary(orc.MODE_FUSED_SHIFTED, d["residual"], d["fn"], d["scale"],
                        d["base"], norm_w, x=d["x"],
                        post_mix=d["post"] if post is None else post,
                        comb=d["comb"] if comb is None else comb, pre_lag=pre_lag)


def test_collapse_one_hot_pre_selects_stream():
    d = synth.make_inputs(3, 64, seed=51)
    for s in range(4):
        pl = np.zeros((3, 4), np.float32)
        pl[:, s] = 1.0
        out = _shifted(d, pl)
        assert np.array_equal(out["layer_input"], out["residual_out"][:, s])


def test_collapse_half_half():
    d = synth.make_inputs(3, 64, seed=52)
    pl = np.zeros((3, 4), np.float32)
    pl[:, 1] = pl[:, 3] = 0.5
    out = _shifted(d, pl)
    cur = B2F(out["residual_out"]).astype(np.float64)
    want = _bf16((0.5 * (cur[:, 1] + cur[:, 3])).astype(np.float32))
    assert np.array_equal(out["layer_input"], want)


def test_unshifted_collapse_uses_own_pre():
    d = synth.make_inputs(3, 64, seed=53)
    out = orc.boundary(orc.MODE_FUSED_UNSHIFTED, d["residual"], d["fn"], d["scale"],
                       d["base"], None, x=d["x"], post_mix=d["post"], comb=d["comb"])
    ref = _shifted(d, out["pre"])                       # the same pre fed as the lag
    assert np.array_equal(out["layer_input"], ref["layer_input"])
    assert np.array_equal(out["residual_out"], ref["residual_out"])


def test_rmsnorm_of_constant_collapse():
    T, H = 3, 64
    d = synth.make_inputs(T, H, seed=54)
    c = np.array([0.75, -2.5, 1.0 / 32], np.float32)
    cb = _bf16(c)
    d["residual"] = np.broadcast_to(cb[:, None, None], (T, 4, H)).copy()
    comb = np.broadcast_to(np.eye(4, dtype=np.float32), (T, 4, 4)).copy()
    post = np.zeros((T, 4), np.float32)
    pl = np.zeros((T, 4), np.float32)
    pl[:, 0] = 1.0
    out = _shifted(d, pl, norm_w=d["norm_w"], comb=comb, post=post)
    cf = B2F(cb).astype(np.float64)
    r = 1.0 / np.sqrt(cf * cf + 1e-6)
    exact = (cf * r)[:, None] * d["norm_w"].astype(np.float64)[None, :]
    want = _bf16(exact.astype(np.float32))
    diff = np.abs(out["layer_input"].astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1
    assert np.allclose(out["rstd_li"], r, rtol=2e-7)


def test_bf16_norm_weight_equals_fp32_of_same_values():
    d = synth.make_inputs(2, 64, seed=55)
    nw16 = _bf16(d["norm_w"])
    a = _shifted(d, d["pre_lag"], norm_w=nw16)
    b = _shifted(d, d["pre_lag"], norm_w=B2F(nw16))
    assert np.array_equal(a["layer_input"], b["layer_input"])


def test_oracle_is_deterministic_and_token_independent():
    d = synth.make_inputs(6, 128, seed=56)
    a = _shifted(d, d["pre_lag"], norm_w=d["norm_w"])
    sub = {k: (v[2:4] if k in ("residual", "x", "post", "comb", "pre_lag") else v)
           for k, v in d.items()}
    b = _shifted(sub, sub["pre_lag"], norm_w=d["norm_w"])
    for k in ("residual_out", "layer_input", "pre", "post", "comb", "mix"):
        assert np.array_equal(a[k][2:4], b[k]), k


# ---------------------------------------------------------------- split-K pre


@pytest.mark.parametrize("weights", [[1.0], [0.5, 0.25, 0.25], [0.5, 0.25, 0.125, 0.125]])
def test_split_k_pre_of_exact_splits_equals_the_boundary(weights):
    """[P] "explaining split-K": the pure path sums the previous GEMM's
    partial mixes and partial sums of squares over the K splits. On a
    small-integer residual the 4H sum of squares is an exact integer, and
    splitting the boundary's own mixes and sum of squares by powers of two
    is exact, so the split-K pre must reproduce pre-only boundary bit for
    bit: same rstd, coefficients, collapse and layer RMSNorm."""
    T, H = 5, 64
    rng = np.random.default_rng(57)
    d = synth.make_inputs(T, H, seed=57)
    d["residual"] = _bf16(rng.integers(-2, 3, size=(T, 4, H)).astype(np.float32))
    ref = orc.boundary(orc.MODE_PRE_ONLY, d["residual"], d["fn"], d["scale"], d["base"],
                       d["norm_w"])
    cur = B2F(d["residual"]).astype(np.float64).reshape(T, -1)
    ssq = (cur * cur).sum(axis=1)                          # exact small integers
    w = np.array(weights, np.float32)
    dot_mix = (w[:, None, None] * ref["mix"][None]).astype(np.float32)
    sqrsum = (w[:, None] * ssq.astype(np.float32)[None]).astype(np.float32)
    assert np.array_equal(dot_mix.astype(np.float64).sum(0), ref["mix"].astype(np.float64))
    out = orc.pre_split_k(d["residual"], dot_mix, sqrsum, d["scale"], d["base"], d["norm_w"])
    for k in ("pre", "post", "comb", "layer_input"):
        assert np.array_equal(out[k], ref[k]), k


def test_split_k_single_split_rstd_and_coefficients():
    """With one split the mixes pass through unchanged and rstd is
    1 / sqrt(sqrsum / 4H + eps), computed here in numpy double; the
    coefficients must then equal the coefficient routine's on those
    values."""
    T, H = 4, 32
    rng = np.random.default_rng(58)
    d = synth.make_inputs(T, H, seed=58)
    dot_mix = rng.normal(0, 3, size=(1, T, 24)).astype(np.float32)
    sqrsum = rng.uniform(10, 500, size=(1, T)).astype(np.float32)
    out = orc.pre_split_k(d["residual"], dot_mix, sqrsum, d["scale"], d["base"], None)
    rstd = (1.0 / np.sqrt(sqrsum[0].astype(np.float64) / (4 * H) + 1e-6)).astype(np.float32)
    pre, post, comb = orc.coefficients(dot_mix[0], rstd, d["scale"], d["base"])
    assert np.array_equal(out["pre"], pre)
    assert np.array_equal(out["post"], post)
    assert np.array_equal(out["comb"], comb)
    # without norm_w the layer input is the raw collapse with this pre
    cur = B2F(d["residual"]).astype(np.float32)
    acc = np.zeros((T, H), np.float32)
    for j in range(4):
        acc = (pre[:, j:j + 1] * cur[:, j] + acc).astype(np.float32)
    want = _bf16(acc)
    diff = np.abs(out["layer_input"].astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1          # numpy's separately rounded multiply-add vs the fma chain


# ---------------------------------------------------------------- regression fixture


def test_oracle_reproduces_the_golden_fixture():
    """tests/golden/tiny_t4_h256_shifted.txt (written by make_golden.py from
    the oracle itself): a regression pin, bit for bit."""
    import os
    import importlib.util
    here = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    spec = importlib.util.spec_from_file_location("make_golden", os.path.join(here, "make_golden.py"))
    mg = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mg)
    want = {}
    with open(os.path.join(here, "tiny_t4_h256_shifted.txt")) as f:
        lines = [l.rstrip("\n") for l in f if not l.startswith("#")]
    for head, body in zip(lines[0::2], lines[1::2]):
        name, dtype, *shape = head.split()
        bits = np.array([int(b, 16) for b in body.split()],
                        np.uint16 if dtype == "uint16" else np.uint32)
        want[name] = bits.view(np.dtype(dtype)).reshape([int(s) for s in shape])
    got = mg.oracle_outputs()
    assert set(got) == set(want)
    for k in got:
        assert np.array_equal(got[k].view(np.uint8), np.ascontiguousarray(want[k]).view(np.uint8)), k


# ---------------------------------------------------------------- orientation, iteration
# count, scale groups and the whole op, against float64 references written
# from the pages ("mhc_boundary": MhcBoundaryKernel.coefficients, sinkhorn,
# col_normalize) in tests/brute64.py, which shares no code with the oracle.

from tests import brute64  # noqa: E402


def _zero_mixer(base, iters, scale=(0.5, 0.5, 0.5), T=1, H=32):
    """Pre-only boundary with fn = 0: every mix is 0, so the logits are the
    base values exactly, whatever rstd and scale are."""
    res = np.zeros((T, 4, H), np.uint16)
    return orc.boundary(orc.MODE_PRE_ONLY, res, np.zeros((24, 4 * H), np.float32),
                        np.asarray(scale, np.float32), np.asarray(base, np.float32), None,
                        params=orc.OracleParams(sinkhorn_iters=iters))


@pytest.mark.parametrize("iters", [1, 2, 20])
def test_comb_orientation_closed_form(iters):
    """Logit (i, k) is base[8 + 4i + k] and comb[i][k] is its entry: with a
    large logit at k = (i + 1) mod 4 of every row i (a non-symmetric
    pattern), softmax and Sinkhorn give nearly that shifted permutation
    matrix, and its transpose gets nearly nothing."""
    base = np.zeros(24, np.float32)
    for i in range(4):
        base[8 + 4 * i + (i + 1) % 4] = 12.0
    c = _zero_mixer(base, iters)["comb"][0].astype(np.float64)
    for i in range(4):
        k = (i + 1) % 4
        assert c[i, k] > 0.999, (i, k, c)
        assert c[k, i] < 1e-3, (k, i, c)                # the transposed entry
        assert abs(c[i].sum() - c[i, k]) < 1e-3


@pytest.mark.parametrize("iters", [1, 2, 5, 20])
def test_softmax_sinkhorn_matches_float64_on_non_symmetric_logits(iters):
    """Random non-symmetric logits (zero mixer, logits = base): the oracle's
    comb equals a float64 row softmax (plus eps), one column normalisation
    and iters - 1 (row, column) normalisations, and pre / post equal
    sigmoid(base) + eps and 2 sigmoid(base). The float64 results one
    iteration fewer or more differ from it well beyond the tolerance (for
    the small counts, before Sinkhorn has converged), so the iteration count
    and the order of the row and column steps are pinned."""
    rng = np.random.default_rng(1000 + iters)
    for trial in range(8):
        base = rng.normal(0.0, 2.0, 24).astype(np.float32)
        out = _zero_mixer(base, iters)
        lg = base[8:].astype(np.float64).reshape(4, 4)
        assert not np.allclose(lg, lg.T)
        want = brute64.softmax_sinkhorn(lg, iters, 1e-6)
        got = out["comb"][0].astype(np.float64)
        assert np.allclose(got, want, rtol=2e-6, atol=1e-9), (iters, trial)
        if iters <= 5:
            for other in (iters - 1, iters + 1):
                if other < 1:
                    continue
                alt = brute64.softmax_sinkhorn(lg, other, 1e-6)
                assert np.max(np.abs(alt - want)) > 1e-4, (iters, other)
            # a softmax over the other index (columns) gives another matrix
            alt_t = brute64.softmax_sinkhorn(lg.T, iters, 1e-6).T
            assert np.max(np.abs(alt_t - want)) > 1e-3
        b = base.astype(np.float64)
        assert np.allclose(out["pre"][0], brute64.sigmoid(b[:4]) + 1e-6, rtol=3e-7, atol=0)
        assert np.allclose(out["post"][0], 2 * brute64.sigmoid(b[4:8]), rtol=3e-7, atol=0)


def test_scale_groups_closed_form():
    """scale[0] multiplies the pre group (mixes 0-3), scale[1] the post group
    (4-7) and scale[2] every comb logit (8-23). A residual with one nonzero
    value (1.0 at stream 0, hidden 0) and a mixer whose column 0 holds
    distinct TF32-exact values a_n makes mix[n] = a_n exactly and the sum of
    squares 1; with scale = (0.25, 1.5, 3.0) every group is then checked
    against its float64 closed form (a swapped group index changes the
    results by orders of magnitude more than the tolerance)."""
    T, H = 1, 32
    K = 4 * H
    res = np.zeros((T, 4, H), np.uint16)
    res[0, 0, 0] = 0x3F80                                  # 1.0
    # |a| <= 0.25 keeps every pre-activation moderate (|v| <= 9 with rstd ~ 11.3
    # and the largest scale), where exp's conditioning leaves the fp32 result
    # within ~1e-6 of the float64 closed form
    a = np.linspace(-0.25, 0.25, 24).astype(np.float32)
    a[8:] = np.random.default_rng(60).permutation(a[8:])   # a non-symmetric logit pattern
    a = orc.tf32_round(a)                                  # exact TF32 values
    assert np.array_equal(brute64.round_tf32(a), a.astype(np.float64))
    fn = np.zeros((24, K), np.float32)
    fn[:, 0] = a
    scale = np.array([0.25, 1.5, 3.0], np.float32)
    base = np.random.default_rng(61).normal(0.0, 0.5, 24).astype(np.float32)
    out = orc.boundary(orc.MODE_PRE_ONLY, res, fn, scale, base, None)
    assert np.array_equal(out["mix"][0], a)
    rstd = 1.0 / np.sqrt(1.0 / K + 1e-6)
    v = a.astype(np.float64) * rstd
    b = base.astype(np.float64)
    pre = brute64.sigmoid(v[:4] * 0.25 + b[:4]) + 1e-6
    post = 2.0 * brute64.sigmoid(v[4:8] * 1.5 + b[4:8])
    comb = brute64.softmax_sinkhorn((v[8:] * 3.0 + b[8:]).reshape(4, 4), 20, 1e-6)
    assert np.allclose(out["pre"][0], pre, rtol=2e-6, atol=0)
    assert np.allclose(out["post"][0], post, rtol=2e-6, atol=0)
    assert np.allclose(out["comb"][0], comb, rtol=1e-5, atol=1e-9)
    # each group away from the others' scales: the check above discriminates
    for wrong in (1.5, 3.0):
        assert not np.allclose(brute64.sigmoid(v[:4] * wrong + b[:4]) + 1e-6, pre, rtol=1e-3)
    for wrong in (0.25, 3.0):
        assert not np.allclose(2.0 * brute64.sigmoid(v[4:8] * wrong + b[4:8]), post, rtol=1e-3)
    for wrong in (0.25, 1.5):
        alt = brute64.softmax_sinkhorn((v[8:] * wrong + b[8:]).reshape(4, 4), 20, 1e-6)
        assert not np.allclose(alt, comb, rtol=1e-3)


MODES_ALL = ("shifted", "unshifted", "pre")


def _oracle_mode(mode, d, iters=20, norm_w=True):
    kw = {}
    if mode != "pre":
        kw = dict(x=d["x"], post_mix=d["post"], comb=d["comb"])
    if mode == "shifted":
        kw["pre_lag"] = d["pre_lag"]
    m = {"pre": orc.MODE_PRE_ONLY, "unshifted": orc.MODE_FUSED_UNSHIFTED,
         "shifted": orc.MODE_FUSED_SHIFTED}[mode]
    return orc.boundary(m, d["residual"], d["fn"], d["scale"], d["base"],
                        d["norm_w"] if norm_w else None,
                        params=orc.OracleParams(sinkhorn_iters=iters), **kw)


def _ulps(a, b):
    def ordered(u):
        v = u.astype(np.int32)
        return np.where(v & 0x8000, -(v & 0x7FFF), v)
    return np.abs(ordered(a) - ordered(b))


@pytest.mark.parametrize("scale", [(0.5, 0.5, 0.5), (0.25, 1.5, 3.0)])
@pytest.mark.parametrize("mode", MODES_ALL)
@pytest.mark.parametrize("norm_w", [True, False])
def test_whole_op_matches_float64_brute_force_on_tiny_workload(mode, norm_w, scale):
    """The whole boundary on the tiny workload (4 tokens, hidden 256, seed 0)
    against the float64 brute force (same steps, double everywhere, bf16
    rounding at the same points): the updated residual and the layer input
    agree bit for bit on this workload (the fp32 chains' rounding never
    moves a bf16 result here; the stress pin below bounds it in general),
    the mixes within 1e-6 of max(|mix|, ||terms||_2), rstd within 1e-6
    relative, and pre / post / comb within 1e-6 relative; with the
    workload's equal scales and with distinct per-group scales."""
    d = synth.workload_inputs("tiny_t4_h256", scale=scale)
    o = _oracle_mode(mode, d, norm_w=norm_w)
    b = brute64.boundary(mode, d, norm_w="f32" if norm_w else None)
    if mode != "pre":
        assert np.array_equal(o["residual_out"], b["residual_out"])
    assert np.array_equal(o["layer_input"], b["layer_input"])
    sc = np.maximum(np.abs(b["mix"]), b["mix_scale"])
    assert np.all(np.abs(o["mix"] - b["mix"]) <= 1e-6 * sc)
    assert np.allclose(o["rstd"], b["rstd"], rtol=1e-6, atol=0)
    assert np.allclose(o["rstd_li"], b["rstd_li"], rtol=1e-6, atol=0)
    for k in ("pre", "post", "comb"):
        assert np.allclose(o[k], b[k], rtol=1e-6, atol=1e-9), k


@pytest.mark.parametrize("iters", [1, 5, 20])
def test_whole_op_stress_against_float64_with_the_chains_error_bound(iters):
    """Stress inputs (residual ~ N(0, 8) with 1 % of entries x100, base ~
    N(0, 4): sigmoid saturates, the update cancels). The updated residual
    is the pages' fp32 flush-to-zero FMA chain rounded to bf16; against the
    exact value rounded once, it may differ by the chain's own error: at
    most 1 bf16 ulp plus 5 fp32 roundings of the chain's largest partial
    magnitude (post*x + sum |comb*res|). Every element is within that, and
    the layer input within 1 ulp; coefficients within 1e-5 relative + 1e-7,
    mixes within 1e-6 of max(|mix|, ||terms||_2)."""
    d = synth.make_inputs(16, 512, seed=4, residual_std=8.0, outlier_frac=0.01,
                          outlier_mult=100.0, base_std=4.0)
    for mode in MODES_ALL:
        o = _oracle_mode(mode, d, iters=iters)
        b = brute64.boundary(mode, d, iters=iters)
        if mode != "pre":
            res = brute64.from_bits(d["residual"])
            x = brute64.from_bits(d["x"])
            mag = (np.abs(d["post"].astype(np.float64))[:, :, None] * np.abs(x)[:, None, :]
                   + np.einsum("tjs,tjh->tsh", np.abs(d["comb"].astype(np.float64)), np.abs(res)))
            go, gb = brute64.from_bits(o["residual_out"]), brute64.from_bits(b["residual_out"])
            ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(gb), 2.0 ** -126))[1] - 8)
            bound = ulp + 5 * 2.0 ** -24 * mag
            assert np.all(np.abs(go - gb) <= bound), mode
        assert _ulps(o["layer_input"], b["layer_input"]).max() <= 1, mode
        for k in ("pre", "post", "comb"):
            assert np.all(np.abs(o[k] - b[k]) <= 1e-5 * np.abs(b[k]) + 1e-7), (mode, k)
        sc = np.maximum(np.abs(b["mix"]), b["mix_scale"])
        assert np.all(np.abs(o["mix"] - b["mix"]) <= 1e-6 * sc), mode


def test_brute_force_rounding_helpers():
    """The float64 reference's own roundings against library routines: bf16
    against torch's RNE conversion (on float32 inputs, whose float64 value
    is exact), TF32 against the arithmetic rounding above."""
    rng = np.random.default_rng(62)
    f = (rng.standard_normal(50_000) * np.exp(rng.uniform(-20, 20, 50_000))).astype(np.float32)
    assert np.array_equal(brute64.bf16_bits(brute64.round_bf16(f.astype(np.float64))),
                          torch_bf16(f))
    w = f[:5000]
    assert np.array_equal(brute64.round_tf32(w),
                          np.array([tf32_arith(float(v)) for v in w], np.float64))
