"""Tensor-core path of Falcon-3 (regression write averaged over a window of
pairs, chunked through sub-chunk key-space recurrences): parity with the
oracle for windows 2..9, several chunks with a ragged tail, carries in and
out (window ring, carried key, position; bit-exact rings), same-step
pairing, a sequence split across two calls, short calls, long runs of
clamped decay, agreement with the column-parallel recurrence, and sampled
heads of the 4 x 8192 x 12, d = 64, W = 8 workload in the launch
configuration the benchmark times."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import TOL, oracle_full, params_for, rel_err
from workloads import FALCON_3, WINDOW_F3, Workload, make_carry, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def w_f3(W, T=300, B=2, H=2, seed=61, **kw):
    return Workload(f"tc_f3_w{W}", FALCON_3, B, T, H, 64, 64, chunk=64, window=W, seed=seed + W, **kw)


def run(F, w, x, carry=None, T=None, impl=None):
    p = params_for(F, w, T=T, impl=F.FALCON_IMPL_TC if impl is None else impl)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    return o, co


def check(o, co, o_ref, c_ref):
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)


def check_carry(co, c_ref):
    assert np.array_equal(co["k_prev"].cpu().double().numpy(), c_ref["k_prev"])
    assert np.array_equal(co["win_x"].cpu().double().numpy(), c_ref["win_x"])
    assert np.array_equal(co["win_v"].cpu().double().numpy(), c_ref["win_v"])
    assert np.array_equal(co["pos"].cpu().numpy(), c_ref["pos"])


@pytest.mark.parametrize("W", [2, 3, 5, 8, 9])
def test_f3_tc_matches_oracle(F, W):
    w = w_f3(W)
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p) == (F.FALCON_IMPL_TC, 2)
    x = make_inputs(w, device="cuda")
    o, co = run(F, w, x)
    o_ref, c_ref = oracle_full(w, x)
    check(o, co, o_ref, c_ref)
    check_carry(co, c_ref)


@pytest.mark.parametrize("W", [4, 8])
@pytest.mark.parametrize("T", [3, 64, 200])
def test_f3_tc_with_carry(F, W, T):
    w = w_f3(W, T=T, B=2, H=3, seed=71)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 89 + W, torch.tensor([[0, 3, 64], [1, 2, 500]]), device="cuda")
    o, co = run(F, w, x, carry)
    o_ref, c_ref = oracle_full(w, x, carry)
    check(o, co, o_ref, c_ref)
    check_carry(co, c_ref)


@pytest.mark.parametrize("W", [4, 8])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_f3_tc_split_sequence(F, W, pairing):
    w = w_f3(W, T=230, pairing=pairing, seed=81)
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    T1 = 97
    x1 = {k: v[:, :T1].contiguous() for k, v in x.items()}
    x2 = {k: v[:, T1:].contiguous() for k, v in x.items()}
    o1, c1 = run(F, w, x1, T=T1)
    o2, c2 = run(F, w, x2, c1, T=w.T - T1)
    check(torch.cat([o1, o2], dim=1), c2, o_ref, c_ref)
    check_carry(c2, c_ref)


@pytest.mark.parametrize("T", [1, 2, 15, 16, 17, 63, 65, 127, 128])
def test_f3_tc_short_and_sub_chunk_edges(F, T):
    w = w_f3(8, T=T, B=1, H=3, seed=91)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, seed=43, pos=3, device="cuda")
    o, co = run(F, w, x, carry)
    o_ref, c_ref = oracle_full(w, x, carry)
    check(o, co, o_ref, c_ref)
    check_carry(co, c_ref)


def test_f3_tc_clamped_runs(F):
    w = w_f3(8, T=400, B=1, H=2, seed=13)
    x = make_inputs(w, device="cuda")
    lam = x["lam"].clone()
    lam[:, 20:60] = 1.0     # a clamped run across sub-chunk and chunk ends
    lam[:, 131:147] = 1.0
    lam[:, 200:330] = 1.0   # two whole chunks of clamped decay
    x["lam"] = lam
    o, co = run(F, w, x)
    o_ref, c_ref = oracle_full(w, x)
    assert torch.isfinite(o.float()).all()
    check(o, co, o_ref, c_ref)


def test_f3_tc_agrees_with_scan(F):
    w = w_f3(8, T=513, B=1, H=3, seed=21)
    x = make_inputs(w, device="cuda")
    o1, c1 = run(F, w, x)
    o2, c2 = run(F, w, x, impl=F.FALCON_IMPL_SCAN)
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(c1["S"].cpu().numpy(), c2["S"].cpu().numpy()) <= TOL["bf16"]
    for n in ("k_prev", "win_x", "win_v", "pos"):
        assert torch.equal(c1[n], c2[n]), n


def test_f3_tc_coverage(F):
    """W = 10 (keys of a sub-chunk past 24) and d = 32 leave the tensor-core
    path: AUTO takes the window recurrence or the portable kernel, a forced
    TC is refused."""
    w = w_f3(8)
    p = params_for(F, w.with_(window=10))
    assert F.falcon_chunk_fwd_plan(p)[0] != F.FALCON_IMPL_TC
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd_plan(params_for(F, w.with_(window=10), impl=F.FALCON_IMPL_TC))
    assert e.value.code == -2
    p = params_for(F, w.with_(dk=32, dv=32))
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_SCAN


def test_f3_tc_full_size_sampled_heads(F):
    """Falcon-3, 4 x 8192 x 12 heads, d = 64, W = 8 in one call (the launch the
    benchmark times): sampled heads recomputed by the oracle's recurrence."""
    import oracle
    w = WINDOW_F3
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p) == (F.FALCON_IMPL_TC, 2)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    heads = [(0, 0), (2, 5), (3, 11)]
    xn = {k: v.cpu().double().numpy() for k, v in x.items()}
    o_ref, S_ref = oracle.recurrent_heads(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"],
                                          w.variant, heads, window=w.window)
    for i, (b, h) in enumerate(heads):
        assert rel_err(o[b, :, h].float().cpu().numpy(), o_ref[i]) <= TOL["bf16"], (b, h)
        assert rel_err(co["S"][b, h].cpu().numpy(), S_ref[i]) <= TOL["bf16"], (b, h)
