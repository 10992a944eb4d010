"""ctypes front end of the C oracle (test infrastructure only; see __init__)."""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mhc_oracle.c")
_LIB = os.path.join(_HERE, "libmhc_oracle.so")

MODE_PRE_ONLY = 0
MODE_FUSED_UNSHIFTED = 1
MODE_FUSED_SHIFTED = 2


class _Params(ctypes.Structure):
    _fields_ = [
        ("hc_norm_eps", ctypes.c_float),
        ("hc_pre_eps", ctypes.c_float),
        ("hc_post_mult", ctypes.c_float),
        ("sinkhorn_eps", ctypes.c_float),
        ("norm_eps", ctypes.c_float),
        ("sinkhorn_iters", ctypes.c_int),
    ]


@dataclass
class OracleParams:
    hc_norm_eps: float = 1e-6
    hc_pre_eps: float = 1e-6
    hc_post_mult: float = 2.0
    sinkhorn_eps: float = 1e-6
    norm_eps: float = 1e-6
    sinkhorn_iters: int = 20

    def _c(self) -> _Params:
        return _Params(self.hc_norm_eps, self.hc_pre_eps, self.hc_post_mult,
                       self.sinkhorn_eps, self.norm_eps, int(self.sinkhorn_iters))


def build_oracle(force: bool = False) -> str:
    """Compile mhc_oracle.c into a shared library next to it (gcc, -O2,
    no contraction of a*b+c into fma, IEEE semantics)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off",
           "-fno-fast-math", "-fno-finite-math-only", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build_oracle())
        P = ctypes.c_void_p
        i64 = ctypes.c_int64
        lib.oracle_tf32_split.argtypes = [P, i64, P, P, P]
        lib.oracle_weight_tiles.argtypes = [P, ctypes.c_int, P]
        lib.oracle_post.argtypes = [P, P, P, P, i64, ctypes.c_int, P]
        lib.oracle_boundary.argtypes = (
            [ctypes.c_int] + [P] * 9 + [ctypes.c_int, ctypes.POINTER(_Params), i64,
                                        ctypes.c_int] + [P] * 9)
        lib.oracle_coefficients.argtypes = [P, P, P, P, ctypes.POINTER(_Params), i64,
                                            P, P, P]
        lib.oracle_f32_to_bf16.argtypes = [P, i64, P]
        lib.oracle_tf32_round.argtypes = [P, i64, P]
        lib.oracle_sigmoid.argtypes = [P, i64, P]
        lib.oracle_sinkhorn.argtypes = [P, i64, ctypes.c_int, ctypes.c_float]
        lib.oracle_pre_split_k.argtypes = ([P, P, P, ctypes.c_int, P, P, P, ctypes.c_int,
                                            ctypes.POINTER(_Params), i64, ctypes.c_int]
                                           + [P] * 4)
        _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype)


def f32_to_bf16(f):
    f = _c(f, np.float32)
    out = np.empty(f.shape, np.uint16)
    _load().oracle_f32_to_bf16(_ptr(f), f.size, _ptr(out))
    return out


def tf32_round(w):
    w = _c(w, np.float32)
    out = np.empty_like(w)
    _load().oracle_tf32_round(_ptr(w), w.size, _ptr(out))
    return out


def tf32_split(w):
    """Returns (rounded fp32, hi bf16 bits, lo bf16 bits)."""
    w = _c(w, np.float32)
    r = np.empty_like(w)
    hi = np.empty(w.shape, np.uint16)
    lo = np.empty(w.shape, np.uint16)
    _load().oracle_tf32_split(_ptr(w), w.size, _ptr(r), _ptr(hi), _ptr(lo))
    return r, hi, lo


def weight_tiles(fn, hidden: int):
    """fn [24, 4H] fp32 -> the library's prepared-weight layout (uint16)."""
    fn = _c(fn, np.float32)
    assert fn.shape == (24, 4 * hidden) and hidden % 32 == 0
    out = np.empty(48 * 4 * hidden, np.uint16)
    _load().oracle_weight_tiles(_ptr(fn), hidden, _ptr(out))
    return out


def sigmoid(v):
    v = _c(v, np.float32)
    out = np.empty_like(v)
    _load().oracle_sigmoid(_ptr(v), v.size, _ptr(out))
    return out


def sinkhorn(c, iters: int, eps: float):
    c = np.array(c, dtype=np.float32, copy=True).reshape(-1, 16)
    _load().oracle_sinkhorn(_ptr(c), c.shape[0], int(iters), float(eps))
    return c


def post(x, residual, post_mix, comb):
    """Residual update only: returns residual_out [T, 4, H] (uint16)."""
    residual = _c(residual, np.uint16)
    T, n, H = residual.shape
    out = np.empty_like(residual)
    _load().oracle_post(_ptr(_c(x, np.uint16)), _ptr(residual),
                        _ptr(_c(post_mix, np.float32)), _ptr(_c(comb, np.float32)),
                        T, H, _ptr(out))
    return out


def coefficients(mix, rstd, scale, base, params: OracleParams | None = None):
    params = params or OracleParams()
    mix = _c(mix, np.float32).reshape(-1, 24)
    rstd = _c(rstd, np.float32).reshape(-1)
    T = mix.shape[0]
    pre = np.empty((T, 4), np.float32)
    post_ = np.empty((T, 4), np.float32)
    comb = np.empty((T, 4, 4), np.float32)
    p = params._c()
    _load().oracle_coefficients(_ptr(mix), _ptr(rstd), _ptr(_c(scale, np.float32)),
                                _ptr(_c(base, np.float32)), ctypes.byref(p), T,
                                _ptr(pre), _ptr(post_), _ptr(comb))
    return pre, post_, comb


def pre_split_k(residual, dot_mix, sqrsum, scale, base, norm_w=None,
                params: OracleParams | None = None):
    """Pre from split-K partial mixes dot_mix [S, T, 24] and partial sums of
    squares sqrsum [S, T]. Returns a dict: layer_input (uint16 [T, H]), pre,
    post, comb."""
    params = params or OracleParams()
    residual = _c(residual, np.uint16)
    T, n, H = residual.shape
    assert n == 4
    dot_mix = _c(dot_mix, np.float32)
    sqrsum = _c(sqrsum, np.float32)
    S = dot_mix.shape[0]
    assert dot_mix.shape == (S, T, 24) and sqrsum.shape == (S, T)
    nw_bf16 = 0
    if norm_w is not None:
        if norm_w.dtype == np.uint16:
            nw_bf16 = 1
        else:
            norm_w = _c(norm_w, np.float32)
    out = {"layer_input": np.empty((T, H), np.uint16), "pre": np.empty((T, 4), np.float32),
           "post": np.empty((T, 4), np.float32), "comb": np.empty((T, 4, 4), np.float32)}
    p = params._c()
    _load().oracle_pre_split_k(_ptr(residual), _ptr(dot_mix), _ptr(sqrsum), S,
                               _ptr(_c(scale, np.float32)), _ptr(_c(base, np.float32)),
                               _ptr(norm_w), nw_bf16, ctypes.byref(p), T, H,
                               _ptr(out["layer_input"]), _ptr(out["pre"]), _ptr(out["post"]),
                               _ptr(out["comb"]))
    return out


def boundary(mode: int, residual, fn, scale, base, norm_w=None, *, x=None,
             post_mix=None, comb=None, pre_lag=None,
             params: OracleParams | None = None):
    """The whole boundary over T tokens. Returns a dict of numpy arrays:
    residual_out (modes 1, 2), layer_input, pre, post, comb and diagnostics
    mix, mix_scale, rstd, rstd_li."""
    params = params or OracleParams()
    residual = _c(residual, np.uint16)
    T, n, H = residual.shape
    assert n == 4
    fn = _c(fn, np.float32)
    assert fn.shape == (24, 4 * H)
    nw_bf16 = 0
    if norm_w is not None:
        if norm_w.dtype == np.uint16:
            nw_bf16 = 1
        else:
            norm_w = _c(norm_w, np.float32)
    x = _c(x, np.uint16)
    post_mix = _c(post_mix, np.float32)
    comb = _c(comb, np.float32)
    pre_lag = _c(pre_lag, np.float32)
    if mode != MODE_PRE_ONLY:
        assert x is not None and post_mix is not None and comb is not None
    if mode == MODE_FUSED_SHIFTED:
        assert pre_lag is not None
    out = {
        "residual_out": np.empty_like(residual) if mode != MODE_PRE_ONLY else None,
        "layer_input": np.empty((T, H), np.uint16),
        "pre": np.empty((T, 4), np.float32),
        "post": np.empty((T, 4), np.float32),
        "comb": np.empty((T, 4, 4), np.float32),
        "mix": np.empty((T, 24), np.float32),
        "mix_scale": np.empty((T, 24), np.float32),
        "rstd": np.empty((T,), np.float32),
        "rstd_li": np.empty((T,), np.float32),
    }
    p = params._c()
    _load().oracle_boundary(
        mode, _ptr(x), _ptr(residual), _ptr(post_mix), _ptr(comb), _ptr(pre_lag),
        _ptr(fn), _ptr(_c(scale, np.float32)), _ptr(_c(base, np.float32)),
        _ptr(norm_w), nw_bf16, ctypes.byref(p), T, H,
        _ptr(out["residual_out"]), _ptr(out["layer_input"]), _ptr(out["pre"]),
        _ptr(out["post"]), _ptr(out["comb"]), _ptr(out["mix"]),
        _ptr(out["mix_scale"]), _ptr(out["rstd"]), _ptr(out["rstd_li"]))
    if out["residual_out"] is None:
        del out["residual_out"]
    return out
