"""Thin ctypes binding of libmhc.so (include/mhc.h).

Argument marshalling only: every step of the boundary runs in the library's
CUDA kernels. Tensors are torch CUDA tensors (bf16 tensors travel as their
bit patterns); outputs are allocated with torch when not given; the call is
enqueued on torch's current stream. There is no fallback: if the library is
missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libmhc.so")
_lib = None

MHC_F32, MHC_BF16 = 0, 1
STATUS_NAMES = {0: "MHC_OK", 1: "MHC_ERR_NULL", 2: "MHC_ERR_ALIGN", 3: "MHC_ERR_SHAPE",
                4: "MHC_ERR_UNSUPPORTED", 5: "MHC_ERR_ALIAS", 6: "MHC_ERR_CUDA",
                7: "MHC_ERR_DEVICE_TIMEOUT", 8: "MHC_ERR_WORKSPACE"}

# every entry point include/mhc.h declares
EXPORTS = ("mhc_weight_bytes", "mhc_prepare_weight", "mhc_post", "mhc_workspace_bytes",
           "mhc_pre", "mhc_boundary_fused", "mhc_get_device_status", "mhc_last_timeout_site",
           "mhc_status_string", "mhc_set_wait_timeout_ns", "mhc_debug_unarmed_wait",
           "mhc_plan", "mhc_debug_record_between", "mhc_boundary_fused_noalloc",
           "mhc_debug_rcp_check", "mhc_pre_split_k", "mhc_debug_coef_check", "mhc_plan_cluster",
           "mhc_debug_set_decode_path", "mhc_debug_set_pdl", "mhc_debug_delayed_copy",
           "mhc_debug_launch_count")


class MhcError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


class _Params(ctypes.Structure):
    _fields_ = [("hc_norm_eps", ctypes.c_float), ("hc_pre_eps", ctypes.c_float),
                ("hc_post_mult", ctypes.c_float), ("sinkhorn_eps", ctypes.c_float),
                ("norm_eps", ctypes.c_float), ("sinkhorn_iters", ctypes.c_int),
                ("batch_invariant", ctypes.c_int)]


@dataclass
class Params:
    hc_norm_eps: float = 1e-6
    hc_pre_eps: float = 1e-6
    hc_post_mult: float = 2.0
    sinkhorn_eps: float = 1e-6
    norm_eps: float = 1e-6
    sinkhorn_iters: int = 20
    batch_invariant: bool = False

    def c(self) -> _Params:
        return _Params(self.hc_norm_eps, self.hc_pre_eps, self.hc_post_mult,
                       self.sinkhorn_eps, self.norm_eps, int(self.sinkhorn_iters),
                       int(bool(self.batch_invariant)))


def lib_path() -> str:
    return _LIB_PATH


def load():
    """Load libmhc.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(f"{_LIB_PATH} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(_LIB_PATH)
    P, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    PP = ctypes.POINTER(_Params)
    sig = {
        "mhc_weight_bytes": (sz, [i32]),
        "mhc_prepare_weight": (i32, [P, i32, P, P]),
        "mhc_post": (i32, [P, P, P, P, P, i64, i32, P]),
        "mhc_workspace_bytes": (sz, [i64, i32]),
        "mhc_pre": (i32, [P, P, P, P, P, i32, PP, i64, i32, P, P, P, P, P, sz, P]),
        "mhc_boundary_fused": (i32, [P, P, P, P, P, P, P, P, P, i32, PP, i64, i32,
                                     P, P, P, P, P, P, sz, P]),
        "mhc_boundary_fused_noalloc": (i32, [P, P, P, P, P, P, P, P, P, i32, PP, i64, i32,
                                             P, P, P, P, P, P]),
        "mhc_get_device_status": (i32, [P]),
        "mhc_last_timeout_site": (i32, []),
        "mhc_status_string": (ctypes.c_char_p, [i32]),
        "mhc_set_wait_timeout_ns": (None, [ctypes.c_uint64]),
        "mhc_debug_unarmed_wait": (i32, [P]),
        "mhc_debug_record_between": (None, [P]),
        "mhc_debug_rcp_check": (i32, [ctypes.c_uint32, ctypes.c_uint64, P, P]),
        "mhc_debug_coef_check": (i32, [P, P, P, PP, i32, i64, P, P, P]),
        "mhc_pre_split_k": (i32, [P, P, P, i32, P, P, P, i32, PP, i64, i32, P, P, P, P, P]),
        "mhc_plan": (i32, [i64, i32, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(ctypes.c_int)]),
        "mhc_plan_cluster": (i32, [i64, i32, ctypes.POINTER(ctypes.c_int)]),
        "mhc_debug_set_decode_path": (None, [i32]),
        "mhc_debug_set_pdl": (None, [i32]),
        "mhc_debug_delayed_copy": (i32, [P, P, i64, ctypes.c_uint32, P]),
        "mhc_debug_launch_count": (ctypes.c_uint64, []),
    }
    for name, (res, args) in sig.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != 0:
        raise MhcError(code, where)


def _p(t):
    # plain ints: the argtypes convert them (cheaper than c_void_p objects)
    return None if t is None else t.data_ptr()


# The current stream's raw handle without building a Stream object (the
# public call costs several microseconds per call on some hosts).
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream=None, device=None):
    if stream is not None:
        return stream.cuda_stream
    if _raw_stream is not None:
        idx = device.index if device is not None and device.index is not None \
            else torch.cuda.current_device()
        return _raw_stream(idx)
    return torch.cuda.current_stream().cuda_stream


_DEFAULT_PARAMS_C = None


def _params_c(params):
    """ctypes struct of `params`; the default one is built once."""
    global _DEFAULT_PARAMS_C
    if params is not None:
        return params.c()
    if _DEFAULT_PARAMS_C is None:
        _DEFAULT_PARAMS_C = Params().c()
    return _DEFAULT_PARAMS_C


def _bf16(t: torch.Tensor, name: str):
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")
    return t


def _f32(t: torch.Tensor, name: str):
    if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA float32 tensor")
    return t


def weight_bytes(hidden: int) -> int:
    return int(load().mhc_weight_bytes(hidden))


def workspace_bytes(tokens: int, hidden: int) -> int:
    return int(load().mhc_workspace_bytes(tokens, hidden))


def plan(tokens: int, hidden: int):
    s, w = ctypes.c_int(), ctypes.c_int()
    _check(load().mhc_plan(tokens, hidden, ctypes.byref(s), ctypes.byref(w)), "mhc_plan")
    return s.value, w.value


def plan_cluster(tokens: int, hidden: int) -> int:
    """Cluster size of a shifted call of (tokens, hidden) on the current
    device, or 0 when it takes the slice-parallel streaming kernel."""
    c = ctypes.c_int()
    _check(load().mhc_plan_cluster(tokens, hidden, ctypes.byref(c)), "mhc_plan_cluster")
    return c.value


def mhc_debug_set_decode_path(path: int):
    """0 (the default): the cluster kernel where it is the faster path; 1:
    every later shifted call takes the slice-parallel streaming kernel; 2:
    the cluster kernel wherever it can run."""
    load().mhc_debug_set_decode_path(int(path))


def mhc_debug_set_pdl(enable: bool):
    """Launch the boundary kernels as programmatic dependents (the default)
    or as plain stream kernels."""
    load().mhc_debug_set_pdl(int(bool(enable)))


def mhc_debug_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(load().mhc_debug_launch_count())


def mhc_debug_delayed_copy(src, dst, delay_ns: int, stream=None):
    """dst <- src (bf16, same size) by a kernel that lets the next kernel on
    the stream start at once and writes only after delay_ns."""
    _bf16(src, "src"), _bf16(dst, "dst")
    if src.numel() != dst.numel():
        raise ValueError("src and dst must have the same size")
    _check(load().mhc_debug_delayed_copy(_p(src), _p(dst), src.numel(), int(delay_ns),
                                         _stream(stream, src.device)), "mhc_debug_delayed_copy")


def mhc_prepare_weight(fn: torch.Tensor, out: torch.Tensor | None = None, stream=None):
    """fn [24, 4H] fp32 -> prepared mixer (uint8, mhc_weight_bytes(H) bytes)."""
    _f32(fn, "fn")
    H = fn.shape[1] // 4
    if out is None:
        out = torch.empty(weight_bytes(H), dtype=torch.uint8, device=fn.device)
    _check(load().mhc_prepare_weight(_p(fn), H, _p(out), _stream(stream)), "mhc_prepare_weight")
    return out


def mhc_post(x, residual, post, comb, out=None, stream=None):
    """Residual update: returns residual_out [T, 4, H] bf16 (may be residual)."""
    _bf16(x, "x"), _bf16(residual, "residual"), _f32(post, "post"), _f32(comb, "comb")
    T, n, H = residual.shape
    if out is None:
        out = torch.empty_like(residual)
    _check(load().mhc_post(_p(x), _p(residual), _p(post), _p(comb), _p(out), T, H,
                           _stream(stream)), "mhc_post")
    return out


def _outs(T, H, dev, layer_input, pre_out, post_out, comb_out, workspace):
    if layer_input is None:
        layer_input = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    if pre_out is None:
        pre_out = torch.empty(T, 4, dtype=torch.float32, device=dev)
    if post_out is None:
        post_out = torch.empty(T, 4, dtype=torch.float32, device=dev)
    if comb_out is None:
        comb_out = torch.empty(T, 4, 4, dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = torch.empty(max(workspace_bytes(T, H), 16), dtype=torch.uint8, device=dev)
    return layer_input, pre_out, post_out, comb_out, workspace


def _nw(norm_w):
    if norm_w is None:
        return None, MHC_F32
    if norm_w.dtype == torch.bfloat16:
        return norm_w, MHC_BF16
    return _f32(norm_w, "norm_w"), MHC_F32


def mhc_pre(residual, weight, scale, base, norm_w=None, params: Params | None = None, *,
            layer_input=None, pre_out=None, post_out=None, comb_out=None, workspace=None,
            stream=None):
    """Unshifted pre: returns (layer_input, pre, post, comb)."""
    _bf16(residual, "residual")
    T, n, H = residual.shape
    li, pr, po, cb, ws = _outs(T, H, residual.device, layer_input, pre_out, post_out,
                               comb_out, workspace)
    nw, nwt = _nw(norm_w)
    p = _params_c(params)
    _check(load().mhc_pre(_p(residual), _p(weight), _p(scale), _p(base), _p(nw), nwt,
                          ctypes.byref(p), T, H, _p(li), _p(pr), _p(po), _p(cb), _p(ws),
                          ws.numel() * ws.element_size(), _stream(stream, residual.device)), "mhc_pre")
    return li, pr, po, cb


def mhc_pre_split_k(residual, dot_mix, sqrsum, scale, base, norm_w=None,
                    params: Params | None = None, *, layer_input=None, pre_out=None,
                    post_out=None, comb_out=None, stream=None):
    """Unshifted pre from split-K partial mixes dot_mix [S, T, 24] and partial
    sums of squares sqrsum [S, T]: returns (layer_input, pre, post, comb)."""
    _bf16(residual, "residual"), _f32(dot_mix, "dot_mix"), _f32(sqrsum, "sqrsum")
    T, n, H = residual.shape
    S = dot_mix.shape[0]
    if tuple(dot_mix.shape) != (S, T, 24) or tuple(sqrsum.shape) != (S, T):
        raise ValueError("dot_mix must be [S, T, 24] and sqrsum [S, T]")
    dev = residual.device
    li = layer_input if layer_input is not None else torch.empty(T, H, dtype=torch.bfloat16,
                                                                 device=dev)
    pr = pre_out if pre_out is not None else torch.empty(T, 4, device=dev)
    po = post_out if post_out is not None else torch.empty(T, 4, device=dev)
    cb = comb_out if comb_out is not None else torch.empty(T, 4, 4, device=dev)
    nw, nwt = _nw(norm_w)
    p = _params_c(params)
    _check(load().mhc_pre_split_k(_p(residual), _p(dot_mix), _p(sqrsum), S, _p(scale), _p(base),
                                  _p(nw), nwt, ctypes.byref(p), T, H, _p(li), _p(pr), _p(po),
                                  _p(cb), _stream(stream, residual.device)), "mhc_pre_split_k")
    return li, pr, po, cb


def mhc_boundary_fused(x, residual, post, comb, weight, scale, base, norm_w=None, pre_lag=None,
                       params: Params | None = None, *, residual_out=None, layer_input=None,
                       pre_out=None, post_out=None, comb_out=None, workspace=None, stream=None):
    """Fused post + pre boundary (shifted when pre_lag is given). Returns
    (residual_out, layer_input, pre, post, comb)."""
    _bf16(x, "x"), _bf16(residual, "residual"), _f32(post, "post"), _f32(comb, "comb")
    if pre_lag is not None:
        _f32(pre_lag, "pre_lag")
    T, n, H = residual.shape
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    li, pr, po, cb, ws = _outs(T, H, residual.device, layer_input, pre_out, post_out,
                               comb_out, workspace)
    nw, nwt = _nw(norm_w)
    p = _params_c(params)
    _check(load().mhc_boundary_fused(
        _p(x), _p(residual), _p(post), _p(comb), _p(pre_lag), _p(weight), _p(scale), _p(base),
        _p(nw), nwt, ctypes.byref(p), T, H, _p(residual_out), _p(li), _p(pr), _p(po), _p(cb),
        _p(ws), ws.numel() * ws.element_size(), _stream(stream, residual.device)), "mhc_boundary_fused")
    return residual_out, li, pr, po, cb


def mhc_boundary_fused_noalloc(x, residual, post, comb, weight, scale, base, norm_w=None,
                               pre_lag=None, params: Params | None = None, *,
                               residual_out=None, layer_input=None, pre_out=None,
                               post_out=None, comb_out=None, stream=None):
    """mhc_boundary_fused whose scratch is the library's fixed device array
    (for callers that cannot allocate device memory). Outputs not given are
    allocated here with torch; pass them all to allocate nothing."""
    _bf16(x, "x"), _bf16(residual, "residual"), _f32(post, "post"), _f32(comb, "comb")
    if pre_lag is not None:
        _f32(pre_lag, "pre_lag")
    T, n, H = residual.shape
    if residual_out is None:
        residual_out = torch.empty_like(residual)
    dev = residual.device
    li = layer_input if layer_input is not None else torch.empty(T, H, dtype=torch.bfloat16,
                                                                 device=dev)
    pr = pre_out if pre_out is not None else torch.empty(T, 4, device=dev)
    po = post_out if post_out is not None else torch.empty(T, 4, device=dev)
    cb = comb_out if comb_out is not None else torch.empty(T, 4, 4, device=dev)
    nw, nwt = _nw(norm_w)
    p = _params_c(params)
    _check(load().mhc_boundary_fused_noalloc(
        _p(x), _p(residual), _p(post), _p(comb), _p(pre_lag), _p(weight), _p(scale), _p(base),
        _p(nw), nwt, ctypes.byref(p), T, H, _p(residual_out), _p(li), _p(pr), _p(po), _p(cb),
        _stream(stream, residual.device)), "mhc_boundary_fused_noalloc")
    return residual_out, li, pr, po, cb


def mhc_get_device_status(stream=None) -> int:
    return int(load().mhc_get_device_status(_stream(stream)))


def mhc_last_timeout_site() -> int:
    return int(load().mhc_last_timeout_site())


def mhc_set_wait_timeout_ns(ns: int):
    load().mhc_set_wait_timeout_ns(int(ns))


def mhc_debug_unarmed_wait(stream=None):
    _check(load().mhc_debug_unarmed_wait(_stream(stream)), "mhc_debug_unarmed_wait")


def mhc_debug_coef_check(values, scale, base, hidden: int, params: Params | None = None,
                         stream=None):
    """Coefficients of the tokens of `values` [n, 25] (fp32, CUDA) formed by
    the one-thread and the 16-lane routines: returns (out_thread, out_lanes),
    each [n, 24] (pre 4, post 4, comb 16)."""
    for t in (values, scale, base):
        if t.dtype != torch.float32 or not t.is_cuda or not t.is_contiguous():
            raise ValueError("values, scale and base must be contiguous CUDA float32 tensors")
    n = values.shape[0]
    p = _params_c(params)
    a = torch.empty(n, 24, dtype=torch.float32, device=values.device)
    b = torch.empty(n, 24, dtype=torch.float32, device=values.device)
    _check(load().mhc_debug_coef_check(_p(values), _p(scale), _p(base), ctypes.byref(p),
                                       int(hidden), n, _p(a), _p(b), _stream(stream)),
           "mhc_debug_coef_check")
    return a, b


def mhc_debug_rcp_check(first_bits: int, count: int, stream=None):
    """(number of bit patterns in [first_bits, first_bits + count) whose
    library reciprocal differs from the correctly rounded one, smallest such
    pattern or None)."""
    s = stream if stream is not None else torch.cuda.current_stream()
    res = torch.tensor([0, -1], dtype=torch.int64, device="cuda")
    s.wait_stream(torch.cuda.current_stream())
    _check(load().mhc_debug_rcp_check(first_bits, count, ctypes.c_void_p(res.data_ptr()),
                                      _stream(s)), "mhc_debug_rcp_check")
    s.synchronize()
    n, first = (int(v) for v in res.cpu().tolist())
    return n, (None if n == 0 else first & 0xFFFFFFFF)


def mhc_debug_record_between(event):
    """Record `event` (torch.cuda.Event) between the streaming and finishing
    kernels of this thread's next mhc_pre / mhc_boundary_fused call."""
    load().mhc_debug_record_between(ctypes.c_void_p(event.cuda_event) if event else None)


def mhc_status_string(code: int) -> str:
    return load().mhc_status_string(int(code)).decode()
