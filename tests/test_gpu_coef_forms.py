"""The two forms of the coefficient step agree bit for bit: one thread per
token (the multi-item shifted path and the finishing kernels) and 16 lanes
per token (a single-wave shifted call, where the end of the call waits on
it). The oracle tests pin the one-thread form to the pages' equations; this
pins the other to it, on ordinary, saturating and degenerate inputs and every
Sinkhorn length the workloads use."""
import numpy as np
import pytest
import torch

from manifold_constrained_hyper_gb300 import ops

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from manifold_constrained_hyper_gb300 import build
    build.build()
    ops.load()


def _values(n, seed):
    g = np.random.default_rng(seed)
    v = np.empty((n, 25), np.float32)
    v[:, :24] = g.normal(0.0, 1.0, (n, 24)) * g.choice([0.01, 1.0, 30.0], (n, 1))
    v[:, 24] = g.uniform(0.1, 4.0, n) * 4096          # a 4H sum of squares at H = 1024
    v[: n // 8, :24] = 0.0                             # zero mixes: the base alone decides
    v[n // 8: n // 4, 8:24] = 1.0                      # uniform comb logits
    return v


@pytest.mark.parametrize("iters", [1, 5, 20])
def test_sixteen_lane_coefficients_equal_one_thread_form(iters):
    n = 1001
    dev = torch.device("cuda")
    v = torch.from_numpy(_values(n, 31 + iters)).to(dev)
    scale = torch.tensor([0.5, 0.5, 0.5], dtype=torch.float32, device=dev)
    g = np.random.default_rng(7)
    for sb in (0.1, 4.0):                              # ordinary and saturating sigmoids
        base = torch.from_numpy(g.normal(0.0, sb, 24).astype(np.float32)).to(dev)
        a, b = ops.mhc_debug_coef_check(v, scale, base, 1024, ops.Params(sinkhorn_iters=iters))
        torch.cuda.synchronize()
        assert torch.isfinite(a).all()
        assert torch.equal(a.view(torch.int32), b.view(torch.int32))
