"""Tensor-core path of Falcon-3A (additive write averaged over a window of
pairs): parity with the oracle when forced for several windows, from carries
(window ring, carried key, position), agreement with the portable path, long
runs of clamped decay, and sampled heads of the 4 x 8192 x 12, d = 64, W = 8
workload in the launch configuration the benchmark times."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import TOL, oracle_full, params_for, rel_err
from workloads import FALCON_3A, WINDOW_F3A, Workload, make_carry, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def w_f3a(W, T=300, B=2, H=2, seed=51):
    return Workload(f"tc_f3a_w{W}", FALCON_3A, B, T, H, 64, 64, chunk=64, window=W, seed=seed + W)


@pytest.mark.parametrize("W", [2, 3, 8, 16])
def test_f3a_tc_forced_matches_oracle(F, W):
    w = w_f3a(W)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    assert F.falcon_chunk_fwd_plan(p) == (F.FALCON_IMPL_TC, 2)  # one chain group at this length
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x)
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)
    assert np.array_equal(co["k_prev"].cpu().double().numpy(), c_ref["k_prev"])
    assert np.array_equal(co["win_x"].cpu().double().numpy(), c_ref["win_x"])
    assert np.array_equal(co["win_v"].cpu().double().numpy(), c_ref["win_v"])
    assert np.array_equal(co["pos"].cpu().numpy(), c_ref["pos"])


@pytest.mark.parametrize("W", [4, 8])
@pytest.mark.parametrize("T", [3, 200])
def test_f3a_tc_with_carry(F, W, T):
    w = w_f3a(W, T=T, B=2, H=3)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 79 + W, torch.tensor([[0, 3, 64], [1, 2, 500]]), device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x, carry)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]
    assert rel_err(co["S"].cpu().numpy(), c_ref["S"]) <= TOL["bf16"]
    assert np.array_equal(co["pos"].cpu().numpy(), c_ref["pos"])
    assert np.array_equal(co["win_x"].cpu().double().numpy(), c_ref["win_x"])
    assert np.array_equal(co["win_v"].cpu().double().numpy(), c_ref["win_v"])


def test_f3a_tc_agrees_with_generic(F):
    w = w_f3a(8, T=513, B=1, H=3)
    x = make_inputs(w, device="cuda")
    outs = {}
    for impl in (F.FALCON_IMPL_TC, F.FALCON_IMPL_GENERIC):
        p = params_for(F, w, impl=impl)
        outs[impl] = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    (o1, c1), (o2, c2) = outs[F.FALCON_IMPL_TC], outs[F.FALCON_IMPL_GENERIC]
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(c1["S"].cpu().numpy(), c2["S"].cpu().numpy()) <= TOL["bf16"]


def test_f3a_tc_clamped_runs(F):
    w = w_f3a(8, T=300, B=1, H=2, seed=11)
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


@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_f3a_tc_chain_in_groups(F, pairing):
    """1 x 1650 x 3 heads (26 chunks, the last one ragged) with a carry: few
    heads over many chunks, so the chain runs in groups (three here: 9, 9
    and 8 chunks), each group starting from the state the earlier groups'
    totals give it; every element against the oracle."""
    w = Workload("tc_f3a_groups", FALCON_3A, 1, 1650, 3, 64, 64, chunk=64, window=8, seed=57,
                 pairing=pairing)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 59, torch.tensor([[0, 9, 300]]), device="cuda")
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p) == (F.FALCON_IMPL_TC, 3)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x, carry)
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)
    for n in ("k_prev", "win_x", "win_v"):
        assert np.array_equal(co[n].cpu().double().numpy(), c_ref[n]), n
    assert np.array_equal(co["pos"].cpu().numpy(), c_ref["pos"])


def test_f3a_tc_full_size_sampled_heads(F):
    """Falcon-3A, 4 x 8192 x 12 heads, d = 64, W = 8: sampled heads against
    the oracle."""
    import oracle
    w = WINDOW_F3A
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    heads = [(0, 0), (3, 11)]
    xn = {k: v.cpu().double().numpy() for k, v in x.items()}
    o_ref, S_ref = oracle.recurrent_heads(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"],
                                          w.variant, heads, window=w.window)
    for i, (b, h) in enumerate(heads):
        assert rel_err(o[b, :, h].float().cpu().numpy(), o_ref[i]) <= TOL["bf16"]
        assert rel_err(co["S"][b, h].cpu().numpy(), S_ref[i]) <= TOL["bf16"]
    assert torch.isfinite(o.float()).all()
