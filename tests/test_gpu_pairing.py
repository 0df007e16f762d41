"""Same-step pairing (pairs (k_t, v_t), the ablation of the prefix
alignment) on every GPU path: the portable chunk kernel for all variants,
each tensor-core path forced, carries across calls, chunk then decode, and
the masked-parallel reference, all against the oracle run with the same
pairing."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, oracle_full, params_for, rel_err, to_np
from workloads import (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, Workload,
                       make_carry, make_inputs)

pytestmark = pytest.mark.gpu

ALL = [FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A]


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def w_same(variant, d=64, T=200, B=2, H=2, W=4, dtype="bf16", seed=91):
    return Workload(f"same_v{variant}_d{d}", variant, B, T, H, d, d, chunk=64,
                    window=W if variant in (FALCON_3, FALCON_3A) else 1, dtype=dtype,
                    seed=seed + variant, pairing="same")


def run(F, w, x, carry=None, impl=None, T=None):
    p = params_for(F, w, T=T, impl=impl)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    return o, co


def check(w, o, co, o_ref, c_ref):
    tol = TOL[w.dtype]
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= tol and e_s <= tol, (e_o, e_s)


@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("impl", ["generic", "auto"])
def test_same_step_chunk_matches_oracle(F, variant, impl):
    w = w_same(variant)
    x = make_inputs(w, device="cuda")
    o, co = run(F, w, x, impl=F.FALCON_IMPL_GENERIC if impl == "generic" else None)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref)
    o_p, _ = oracle.recurrent(*(to_np(x)[n] for n in ("q", "k", "v", "beta", "lam")), w.variant,
                              w.window)
    assert rel_err(o_p, o_ref) > 1e-2  # a different method than the prefix alignment


@pytest.mark.parametrize("variant,d,W", [(FALCON_1, 64, 1), (FALCON_1, 128, 1), (FALCON_1A, 64, 1),
                                         (FALCON_1A, 128, 1), (FALCON_2, 64, 1), (FALCON_2, 128, 1),
                                         (FALCON_2A, 128, 1), (FALCON_3A, 64, 8)])
def test_same_step_tensor_core_paths(F, variant, d, W):
    w = w_same(variant, d=d, T=300, W=W)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    o, co = run(F, w, x, impl=F.FALCON_IMPL_TC)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref)


@pytest.mark.parametrize("variant", ALL)
def test_same_step_carry_round_trip(F, variant):
    w = w_same(variant, T=230)
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    T1 = 97
    xa = {k: v[:, :T1].contiguous() for k, v in x.items()}
    xb = {k: v[:, T1:].contiguous() for k, v in x.items()}
    oa, ca = run(F, w, xa, T=T1)
    ob, cb = run(F, w, xb, carry=ca, T=w.T - T1)
    check(w, torch.cat([oa, ob], 1), cb, o_ref, c_ref)
    assert np.array_equal(cb["pos"].cpu().numpy(), c_ref["pos"])
    if "win_x" in c_ref:
        assert np.array_equal(cb["win_x"].cpu().double().numpy(), c_ref["win_x"])
        assert np.array_equal(cb["win_v"].cpu().double().numpy(), c_ref["win_v"])


@pytest.mark.parametrize("variant", ALL)
def test_same_step_synthetic_carry(F, variant):
    w = w_same(variant, T=150, B=2, H=3)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 93, torch.tensor([[0, 1, 5], [2, 40, 3]]), device="cuda")
    o, co = run(F, w, x, carry=carry)
    o_ref, c_ref = oracle_full(w, x, carry)
    check(w, o, co, o_ref, c_ref)


@pytest.mark.parametrize("variant", ALL)
def test_same_step_chunk_then_decode(F, variant):
    w = w_same(variant, T=131)
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    T0 = w.T - 1
    xa = {k: v[:, :T0].contiguous() for k, v in x.items()}
    oa, ca = run(F, w, xa, T=T0)
    p1 = params_for(F, w, T=1)
    o1 = torch.empty((w.B, 1, w.H, w.dv), dtype=x["q"].dtype, device="cuda")
    F.falcon_recurrent_step(p1, *(x[n][:, T0:].contiguous() for n in ("q", "k", "v", "beta", "lam")),
                            ca, o1)
    torch.cuda.synchronize()
    check(w, torch.cat([oa, o1], 1), ca, o_ref, c_ref)


@pytest.mark.parametrize("variant", ALL)
def test_same_step_masked_parallel(F, variant):
    w = w_same(variant, T=96, d=32, W=3, dtype="f32")
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    o, S = F.masked_parallel(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.masked_parallel(*(to_np(x)[n] for n in ("q", "k", "v", "beta", "lam")),
                                          w.variant, w.window, pairing="same")
    assert rel_err(o.cpu().numpy(), o_ref) <= 1e-4
    assert rel_err(S.cpu().numpy(), S_ref) <= 1e-4
