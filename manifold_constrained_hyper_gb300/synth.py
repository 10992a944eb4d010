"""Seeded synthetic inputs for the mHC boundary (no arithmetic of the method).

The pages name no dataset; these generators make the tensors of the boundary
with the shapes and value distributions of the workloads it is quoted on:

* residual ``[T, 4, H]`` bf16 ~ N(0, residual_std), optionally with a fraction
  of entries multiplied by ``outlier_mult`` (the stress workload);
* layer output ``x [T, H]`` bf16 ~ N(0, 1);
* previous boundary's ``post [T, 4]`` ~ U(0, 2);
* previous boundary's ``comb [T, 4, 4]``: a random doubly stochastic matrix,
  drawn as a random convex combination of the 24 permutation matrices of
  size 4 (Birkhoff), so its rows and columns sum to 1;
* previous boundary's ``pre_lag [T, 4]`` = 1e-6 + U(0, 1);
* mixer ``fn [24, 4H]`` fp32 ~ N(0, 1/sqrt(4H)) (standard deviation);
* ``scale = (0.5, 0.5, 0.5)`` unless given (the per-group scales of pre,
  post and comb), ``base [24]`` ~ N(0, base_std), ``norm_w [H]`` fp32 =
  1 + N(0, 0.02).

Everything comes from one ``torch.Generator('cpu')`` seeded with ``seed`` and
is returned as numpy arrays (bf16 as ``uint16`` bit patterns) so that the CUDA
path and the CPU oracle consume the very same bytes.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import torch

# Workloads (shapes, seeds and distributions); names say what they are.
WORKLOADS = {
    "tiny_t4_h256": dict(T=4, H=256, seed=0),
    "mid_t512_h7168": dict(T=512, H=7168, seed=2),
    "prefill_t8192_h7168": dict(T=8192, H=7168, seed=3),
    "stress_t1024_h4096": dict(T=1024, H=4096, seed=4, residual_std=8.0,
                               outlier_frac=0.01, outlier_mult=100.0, base_std=4.0),
}
DECODE_TOKENS = (1, 2, 4, 8, 16, 32, 64)
DECODE_HIDDEN = 7168


def decode_workload(T: int) -> dict:
    return dict(T=T, H=DECODE_HIDDEN, seed=1000 + T)


_PERMS = np.array([np.eye(4, dtype=np.float64)[list(p)]
                   for p in itertools.permutations(range(4))])  # [24, 4, 4]


def _bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()


def make_inputs(T: int, H: int, seed: int, *, residual_std: float = 1.0,
                outlier_frac: float = 0.0, outlier_mult: float = 100.0,
                base_std: float = 0.1, with_fn: bool = True,
                scale=(0.5, 0.5, 0.5)) -> dict:
    """All inputs of one boundary call (see the module docstring)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    res = torch.randn(T, 4, H, generator=g, dtype=torch.float32) * residual_std
    if outlier_frac > 0.0 and res.numel() > 0:
        mask = torch.rand(T, 4, H, generator=g) < outlier_frac
        res = torch.where(mask, res * outlier_mult, res)
    x = torch.randn(T, H, generator=g, dtype=torch.float32)
    return _finish(g, T, H, res, x, base_std, with_fn, scale)


def make_inputs_device(T: int, H: int, seed: int, device, *, residual_std: float = 1.0,
                       outlier_frac: float = 0.0, outlier_mult: float = 100.0,
                       base_std: float = 0.1, scale=(0.5, 0.5, 0.5)) -> dict:
    """Same recipe for large workloads: residual and x are drawn on `device`
    by a generator seeded with `seed` and stay there as bf16 tensors
    (``residual_dev``, ``x_dev``); the small tensors come from a CPU generator
    seeded with ``seed + 1`` as numpy arrays. Rows needed on the host are
    copied back by the caller."""
    gd = torch.Generator(device).manual_seed(int(seed))
    res = torch.randn(T, 4, H, generator=gd, dtype=torch.float32, device=device)
    res.mul_(residual_std)
    if outlier_frac > 0.0 and res.numel() > 0:
        mask = torch.rand(T, 4, H, generator=gd, device=device) < outlier_frac
        res = torch.where(mask, res * outlier_mult, res)
    x = torch.randn(T, H, generator=gd, dtype=torch.float32, device=device)
    g = torch.Generator("cpu").manual_seed(int(seed) + 1)
    out = _finish(g, T, H, None, None, base_std, True, scale)
    out["residual_dev"] = res.to(torch.bfloat16)
    del res
    out["x_dev"] = x.to(torch.bfloat16)
    return out


def _finish(g, T, H, res, x, base_std, with_fn, scale):
    post = torch.rand(T, 4, generator=g, dtype=torch.float32) * 2.0
    # Birkhoff: convex weights from normalised exponential draws
    e = -torch.log(torch.rand(T, 24, generator=g, dtype=torch.float64).clamp_min(1e-300))
    lam = (e / e.sum(dim=1, keepdim=True)).numpy()
    comb = np.einsum("tp,pij->tij", lam, _PERMS).astype(np.float32)
    pre_lag = (torch.rand(T, 4, generator=g, dtype=torch.float32) + 1e-6).numpy()
    out = dict(post=post.numpy(), comb=comb, pre_lag=pre_lag)
    if res is not None:
        out["residual"] = _bf16_bits(res)
        out["x"] = _bf16_bits(x)
    if with_fn:
        K = 4 * H
        out["fn"] = (torch.randn(24, K, generator=g, dtype=torch.float32)
                     * (1.0 / np.sqrt(K))).numpy()
        out["scale"] = np.array(scale, np.float32).reshape(3)
        out["base"] = (torch.randn(24, generator=g, dtype=torch.float32) * base_std).numpy()
        out["norm_w"] = (1.0 + torch.randn(H, generator=g, dtype=torch.float32) * 0.02).numpy()
    return out


def workload_inputs(name: str, **overrides) -> dict:
    cfg = dict(WORKLOADS[name])
    cfg.update(overrides)
    return make_inputs(**cfg)


def make_split_k_inputs(T: int, H: int, S: int, seed: int, **kw) -> dict:
    """Inputs of one split-K pre call: make_inputs' tensors plus the previous
    GEMM's outputs stood in for by seeded random numbers: dot_mix [S, T, 24]
    ~ N(0, 1 / sqrt(S)) (the mixes of N(0, 1) residuals with fn ~ N(0,
    1 / sqrt(4H)) are about N(0, 1)), and sqrsum [S, T] ~ (4H / S) * U(0.8,
    1.2) (positive, summing to about 4H)."""
    d = make_inputs(T, H, seed, **kw)
    g = torch.Generator("cpu").manual_seed(int(seed) + 7)
    d["dot_mix"] = (torch.randn(S, T, 24, generator=g) / math.sqrt(S)).numpy().astype(np.float32)
    d["sqrsum"] = ((4.0 * H / S) * (0.8 + 0.4 * torch.rand(S, T, generator=g))).numpy().astype(
        np.float32)
    return d


def bf16_bits_to_float(a: np.ndarray) -> np.ndarray:
    """uint16 bf16 bit patterns -> float32 values (exact widening)."""
    return (a.astype(np.uint32) << 16).view(np.float32)
