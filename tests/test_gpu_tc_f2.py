"""Tensor-core path of Falcon-2 / Falcon-2A (NLMS step per value channel):
parity with the oracle when forced, with carries, agreement with the portable
path, and sampled heads of the 4 x 4096 x 16, d = 128 workload in the launch
configuration the benchmark times."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import TOL, oracle_full, params_for, rel_err
from workloads import FALCON_2, FALCON_2A, PERCH_F2, Workload, make_carry, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def w_f2(variant, d=64, T=300, B=2, H=2, seed=41):
    return Workload(f"tc_f2_v{variant}_d{d}", variant, B, T, H, d, d, chunk=64, seed=seed + variant)


@pytest.mark.parametrize("variant", [FALCON_2, FALCON_2A])
@pytest.mark.parametrize("d", [64, 128])
def test_f2_tc_forced_matches_oracle(F, variant, d):
    w = w_f2(variant, d=d)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    assert F.falcon_chunk_fwd_plan(p) == (F.FALCON_IMPL_TC, 1)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x)
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)
    assert torch.equal(co["k_prev"].cpu(), x["k"][:, -1].cpu())
    assert torch.all(co["pos"].cpu() == w.T)


@pytest.mark.parametrize("variant", [FALCON_2, FALCON_2A])
@pytest.mark.parametrize("d", [64, 128])
def test_f2_tc_with_carry(F, variant, d):
    w = w_f2(variant, d=d, T=200, B=2, H=3)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 78, torch.tensor([[0, 3, 64], [1, 2, 500]]), device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x, carry)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]
    assert rel_err(co["S"].cpu().numpy(), c_ref["S"]) <= TOL["bf16"]
    assert np.array_equal(co["pos"].cpu().numpy(), c_ref["pos"])


@pytest.mark.parametrize("variant", [FALCON_2, FALCON_2A])
def test_f2_tc_agrees_with_generic(F, variant):
    w = w_f2(variant, d=128, T=257, B=1, H=2)
    x = make_inputs(w, device="cuda")
    outs = {}
    for impl in (F.FALCON_IMPL_TC, F.FALCON_IMPL_GENERIC):
        p = params_for(F, w, impl=impl)
        outs[impl] = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    (o1, c1), (o2, c2) = outs[F.FALCON_IMPL_TC], outs[F.FALCON_IMPL_GENERIC]
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(c1["S"].cpu().numpy(), c2["S"].cpu().numpy()) <= TOL["bf16"]


def test_f2_tc_clamped_runs(F):
    """Long runs of clamped decay: the in-block decay ratios underflow and the
    kernel falls back to exact exponentials."""
    w = w_f2(FALCON_2, d=64, T=300, B=1, H=2, seed=9)
    x = make_inputs(w, device="cuda")
    lam = x["lam"].clone()
    lam[:, 20:60] = 1.0
    lam[:, 131:147] = 1.0
    x["lam"] = lam
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x)
    assert torch.isfinite(o.float()).all()
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]
    assert rel_err(co["S"].cpu().numpy(), c_ref["S"]) <= TOL["bf16"]


def test_f2_tc_full_size_sampled_heads(F):
    """Falcon-2, 4 x 4096 x 16 heads, d = 128, bf16, beta per channel: sampled
    heads against the oracle."""
    import oracle
    w = PERCH_F2
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    heads = [(0, 0), (2, 9), (3, 15)]
    xn = {k: v.cpu().double().numpy() for k, v in x.items()}
    o_ref, S_ref = oracle.recurrent_heads(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"],
                                          w.variant, heads)
    for i, (b, h) in enumerate(heads):
        assert rel_err(o[b, :, h].float().cpu().numpy(), o_ref[i]) <= TOL["bf16"]
        assert rel_err(co["S"][b, h].cpu().numpy(), S_ref[i]) <= TOL["bf16"]
    assert torch.isfinite(o.float()).all()
