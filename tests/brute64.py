"""A float64 brute force of the mHC boundary, for pinning the CPU oracle.

Independent of the oracle (numpy, no shared code): every step is written from
the pages' definitions with the arithmetic done in float64, and the bf16
roundings kept at the points the pages put them (the updated residual, the
collapse, the layer input). The TF32 rounding of the mixer is done by
arithmetic on the value (round to 11 significant bits, ties away from zero),
not by the bit trick the oracle uses. Page references: "mhc_boundary" is the
vLLM DeepSeek-V4.1 shifted mHC boundary API page (residual_update,
MhcBoundaryKernel.coefficients / sinkhorn / col_normalize, lagged_collapse,
layer_input_words); "pre study" is "The Hyper Connection Preprocessing GPU
Kernel Study" ("square sum and RMSNorm", "computing A_l / B_l / C_l",
"computing layer_input").
"""
from __future__ import annotations

import numpy as np


def round_bf16(v) -> np.ndarray:
    """float64 -> nearest bf16 value (8 significant bits, ties to even), as
    float64. Values of magnitude below 2^-126 are flushed to zero (the
    update chain flushes subnormals; the data never reach them elsewhere)."""
    v = np.asarray(v, np.float64)
    out = np.zeros_like(v)
    nz = np.abs(v) >= 2.0 ** -126
    m, e = np.frexp(v[nz])                       # v = m 2^e, 0.5 <= |m| < 1
    q = np.ldexp(m, 8)                           # 8 significant bits above the point
    out[nz] = np.ldexp(np.rint(q), e - 8)        # rint: ties to even, exact scaling
    return out


def bf16_bits(v64: np.ndarray) -> np.ndarray:
    """bf16-representable float64 values -> uint16 bit patterns."""
    f = np.asarray(v64, np.float64).astype(np.float32)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def from_bits(u: np.ndarray) -> np.ndarray:
    return (np.asarray(u).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def round_tf32(w) -> np.ndarray:
    """Round to 11 significant bits (TF32), ties away from zero, by arithmetic."""
    w = np.asarray(w, np.float64)
    out = np.zeros_like(w)
    nz = w != 0
    m, e = np.frexp(np.abs(w[nz]))
    q = np.ldexp(m, 11)
    out[nz] = np.sign(w[nz]) * np.ldexp(np.floor(q + 0.5), e - 11)
    return out


def sigmoid(v):
    return 1.0 / (1.0 + np.exp(-np.asarray(v, np.float64)))


def softmax_sinkhorn(logits: np.ndarray, iters: int, eps: float) -> np.ndarray:
    """logits [..., 4, 4] (row i, column k): row softmax plus eps, one column
    normalisation, then iters - 1 times a row and a column normalisation,
    each dividing by (sum + eps)."""
    lg = np.asarray(logits, np.float64)
    e = np.exp(lg - lg.max(axis=-1, keepdims=True))
    c = e / e.sum(axis=-1, keepdims=True) + eps
    c = c / (c.sum(axis=-2, keepdims=True) + eps)
    for _ in range(iters - 1):
        c = c / (c.sum(axis=-1, keepdims=True) + eps)
        c = c / (c.sum(axis=-2, keepdims=True) + eps)
    return c


def boundary(mode: str, d: dict, scale=None, iters: int = 20, hc_norm_eps: float = 1e-6,
             pre_eps: float = 1e-6, post_mult: float = 2.0, sk_eps: float = 1e-6,
             norm_eps: float = 1e-6, norm_w="f32") -> dict:
    """The whole boundary over the tokens of `d` (synth inputs). mode: "pre"
    (no update), "unshifted" or "shifted" (collapse with d["pre_lag"])."""
    res = from_bits(d["residual"])                              # [T, 4, H]
    T, n, H = res.shape
    K = n * H
    if mode == "pre":
        cur = res
    else:
        x = from_bits(d["x"])                                   # [T, H]
        post = d["post"].astype(np.float64)                     # [T, 4]
        comb = d["comb"].astype(np.float64)                     # [T, j, s]
        exact = post[:, :, None] * x[:, None, :] + np.einsum("tjs,tjh->tsh", comb, res)
        cur = round_bf16(exact)
    flat = cur.reshape(T, K)
    ssq = (flat * flat).sum(axis=1)
    rstd = 1.0 / np.sqrt(ssq / K + hc_norm_eps)
    w = round_tf32(d["fn"])                                     # [24, K]
    mix = flat @ w.T                                            # [T, 24]
    mix_scale = np.sqrt((flat * flat) @ (w * w).T)             # ||(w_k x_k)_k||_2
    s = np.asarray(d["scale"] if scale is None else scale, np.float64)
    b = d["base"].astype(np.float64)
    v = mix * rstd[:, None]
    pre = sigmoid(v[:, 0:4] * s[0] + b[0:4]) + pre_eps
    post_o = sigmoid(v[:, 4:8] * s[1] + b[4:8]) * post_mult
    logits = (v[:, 8:24] * s[2] + b[8:24]).reshape(T, 4, 4)
    comb_o = softmax_sinkhorn(logits, iters, sk_eps)
    pc = d["pre_lag"].astype(np.float64) if mode == "shifted" else pre
    li = round_bf16(np.einsum("tj,tjh->th", pc, cur))
    rstd_li = 1.0 / np.sqrt((li * li).sum(axis=1) / H + norm_eps)
    if norm_w is None:
        out = li
    else:
        nw = d["norm_w"].astype(np.float64)
        if norm_w == "bf16":
            nw = round_bf16(nw)
        out = round_bf16(li * rstd_li[:, None] * nw[None, :])
    r = dict(layer_input=bf16_bits(out), pre=pre, post=post_o, comb=comb_o, mix=mix,
             mix_scale=mix_scale, rstd=rstd, rstd_li=rstd_li, collapse=li)
    if mode != "pre":
        r["residual_out"] = bf16_bits(cur)
    return r
