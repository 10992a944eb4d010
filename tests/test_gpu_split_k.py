"""GPU parity of the split-K pre ("The Hyper Connection Preprocessing GPU
Kernel Study", the pure path) against the oracle: the GPU sums the splits in
split order in fp32, the oracle in double, so the coefficients are compared
at 1e-5 relative and the layer input at 1 bf16 ulp against the oracle's
collapse of the GPU's own pre (and 99.9 % within 1 ulp independently)."""
import numpy as np
import pytest
import torch

import oracle as orc
from manifold_constrained_hyper_gb300 import ops, synth
from tests.mhc_testlib import bf16_ulp_diff, dev_bf16, dev_f32, oracle_layer_input_given_pre

pytestmark = pytest.mark.gpu


def run_split_k(d, norm="f32"):
    nw = None
    if norm == "f32":
        nw = dev_f32(d["norm_w"])
    elif norm == "bf16":
        nw = dev_bf16(orc.f32_to_bf16(d["norm_w"]))
    li, pr, po, cb = ops.mhc_pre_split_k(dev_bf16(d["residual"]), dev_f32(d["dot_mix"]),
                                         dev_f32(d["sqrsum"]), dev_f32(d["scale"]),
                                         dev_f32(d["base"]), nw)
    torch.cuda.synchronize()
    return dict(layer_input=li.view(torch.int16).cpu().numpy().view(np.uint16),
                pre=pr.cpu().numpy(), post=po.cpu().numpy(), comb=cb.cpu().numpy())


def check(d, g, norm="f32"):
    nw = {"f32": d["norm_w"], "bf16": orc.f32_to_bf16(d["norm_w"]), None: None}[norm]
    o = orc.pre_split_k(d["residual"], d["dot_mix"], d["sqrsum"], d["scale"], d["base"], nw)
    for k in ("pre", "post", "comb"):
        np.testing.assert_allclose(g[k], o[k], rtol=1e-5, atol=1e-7, err_msg=k)
    own = oracle_layer_input_given_pre("pre", d, g["pre"], norm=norm)
    assert bf16_ulp_diff(g["layer_input"], own).max() <= 1
    ind = bf16_ulp_diff(g["layer_input"], o["layer_input"])
    assert (ind <= 1).mean() >= 0.999


@pytest.mark.parametrize("S", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("T,H", [(1, 7168), (37, 256), (129, 4096), (300, 7168), (1024, 512)])
def test_split_k_pre_parity(S, T, H):
    d = synth.make_split_k_inputs(T, H, S, seed=700 + T + S)
    check(d, run_split_k(d))


@pytest.mark.parametrize("norm", ["bf16", None])
def test_split_k_pre_norm_variants(norm):
    d = synth.make_split_k_inputs(70, 1024, 4, seed=777)
    check(d, run_split_k(d, norm), norm)


def test_split_k_pre_more_splits_than_the_page_and_deterministic():
    d = synth.make_split_k_inputs(300, 512, 37, seed=778)
    a = run_split_k(d)
    check(d, a)
    b = run_split_k(d)
    for k in a:
        assert np.array_equal(a[k], b[k]), k


def test_split_k_pre_at_hidden_7168_4096_tokens_sampled():
    T, H, S = 4096, 7168, 4
    d = synth.make_split_k_inputs(T, H, S, seed=779)
    g = run_split_k(d)
    rows = np.unique(np.concatenate([[0, 31, 32, T - 1], np.random.default_rng(4096).integers(0, T, 24)]))
    sub = dict(d, residual=d["residual"][rows], dot_mix=d["dot_mix"][:, rows],
               sqrsum=d["sqrsum"][:, rows])
    check(sub, {k: v[rows] for k, v in g.items()})
