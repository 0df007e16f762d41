"""Backward pass (falcon_backward through the C ABI) against the backward
oracle (torch fp64 autodiff of the one-pair recurrence; the window variants
and d = 128 are in test_gpu_backward_window.py): every gradient
element by element, for Falcon-1/1A/2/2A, both pairings, bf16 and fp32,
d = 32 and 64, carried state / key / positions, clamped decays, the empty
and one-step sequences, block boundaries (64 steps) and a ragged tail; and,
at the full 8 x 2048 x 12 d64 size and over 16384 steps (256 chunks), sampled
heads computed one by one."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import params_for, rel_err, to_np
from workloads import (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, Workload,
                       make_carry, make_cotangents, make_inputs)

pytestmark = pytest.mark.gpu

ONE_PAIR = [FALCON_1, FALCON_1A, FALCON_2, FALCON_2A]
# dq, dk, dv are stored in the dtype (bf16 rounding 2^-9 relative, plus fp32
# accumulation over the sequence); dbeta, dlam, dS_in are fp32 outputs of fp32
# arithmetic on the same (dtype-rounded) inputs the oracle sees in fp64.
TOL_D = {"bf16": 2e-2, "f32": 1e-3}
TOL_F32 = {"bf16": 2e-3, "f32": 1e-3}


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def wl(variant, d=64, T=200, B=2, H=3, dtype="bf16", pairing="prefix", seed=301, **kw):
    return Workload(f"bwd_v{variant}_d{d}", variant, B, T, H, d, d, chunk=64, dtype=dtype,
                    seed=seed + variant, pairing=pairing, **kw)


def run_both(F, w, carry=None, with_dS=True, cot_seed=7):
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, cot_seed, device="cuda", with_dS=with_dS)
    p = params_for(F, w)
    g = F.backward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"], c["dS_final"], carry)
    torch.cuda.synchronize()
    xn = to_np(x)
    cn = to_np({k: v for k, v in c.items() if v is not None})
    ref = oracle.recurrent_vjp(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"], w.variant,
                               cn["dO"], cn.get("dS_final"), w.eps, w.eps_gamma,
                               carry=to_np(carry), pairing=w.pairing)
    return g, ref


def check(w, g, ref, names=("dq", "dk", "dv", "dbeta", "dlam")):
    errs = {}
    for n in names:
        tol = TOL_D[w.dtype] if n in ("dq", "dk", "dv", "dk_prev") else TOL_F32[w.dtype]
        e = rel_err(g[n].double().cpu().numpy(), ref[n])
        errs[n] = e
        assert e <= tol, (n, e, errs)
    return errs


@pytest.mark.parametrize("variant", ONE_PAIR)
@pytest.mark.parametrize("pairing", ["prefix", "same"])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_backward_matches_oracle(F, variant, pairing, dtype):
    w = wl(variant, dtype=dtype, pairing=pairing)
    g, ref = run_both(F, w)
    check(w, g, ref)
    assert torch.isfinite(g["dS_in"]).all()
    if pairing == "same":
        assert float(g["dk_prev"].abs().max()) == 0.0


@pytest.mark.parametrize("variant", ONE_PAIR)
@pytest.mark.parametrize("d", [32, 64])
def test_backward_with_carry(F, variant, d):
    w = wl(variant, d=d, T=150, seed=411)
    pos = torch.tensor([[0, 1, 57], [300, 2, 0]], dtype=torch.int64)
    carry = make_carry(w, seed=12, pos=pos, device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=("dq", "dk", "dv", "dbeta", "dlam", "dS_in", "dk_prev"))


@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_backward_carry_same_step_and_f2(F, pairing):
    w = wl(FALCON_2, T=97, pairing=pairing, seed=521)
    carry = make_carry(w, seed=13, pos=5, device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=("dq", "dk", "dv", "dbeta", "dlam", "dS_in", "dk_prev"))


@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 128, 129])
def test_backward_block_edges(F, T):
    w = wl(FALCON_1, T=T, B=1, H=2, seed=601)
    carry = make_carry(w, seed=14, pos=3, device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=("dq", "dk", "dv", "dbeta", "dlam", "dS_in", "dk_prev"))


def test_backward_empty_sequence(F):
    w = wl(FALCON_1, T=0, B=2, H=2)
    carry = make_carry(w, seed=15, pos=4, device="cuda")
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 3, device="cuda")
    g = F.backward(params_for(F, w), x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"],
                   c["dS_final"], carry)
    torch.cuda.synchronize()
    assert torch.equal(g["dS_in"], c["dS_final"])
    assert float(g["dk_prev"].float().abs().max()) == 0.0


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_2A])
def test_backward_clamped_decay(F, variant):
    w = wl(variant, T=180, force_zero_gamma=0.2, gamma_mu=-1.0, gamma_sd=3.0, seed=701)
    g, ref = run_both(F, w)
    check(w, g, ref)
    lam = make_inputs(w)["lam"]
    clamped = (1.0 - lam) < w.eps_gamma
    assert clamped.any()
    assert float(g["dlam"].cpu()[clamped].abs().max()) == 0.0


def test_backward_rejects_window_past_the_limit(F):
    """Falcon-3/3A are covered up to the window the window kernel's shared
    memory holds (34 at d = 128); a wider one is refused on the host."""
    w = wl(FALCON_3, d=128, T=10, window=35)
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 1, device="cuda")
    with pytest.raises(F.FalconError) as e:
        F.backward(params_for(F, w), x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"], None)
    assert e.value.code == -2


def test_backward_long_sequence_sampled_head(F):
    """Falcon-1, 1 x 16384 x 2 heads, d = 64, bf16: 256 chunks, so the chains
    carry their products of split-bf16 operands (transition and state) through
    256 steps; one head is recomputed by the oracle, the gradient of the
    (zero) start state included."""
    w = wl(FALCON_1, T=16384, B=1, H=2, seed=811)
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 11, device="cuda")
    g = F.backward(params_for(F, w), x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"],
                   c["dS_final"])
    torch.cuda.synchronize()
    xn = to_np(x)
    cn = to_np(c)
    h = 1
    sl = lambda a: a[:, :, h:h + 1]
    ref = oracle.recurrent_vjp(sl(xn["q"]), sl(xn["k"]), sl(xn["v"]), sl(xn["beta"]), sl(xn["lam"]),
                               w.variant, sl(cn["dO"]), cn["dS_final"][:, h:h + 1], w.eps, w.eps_gamma,
                               carry={"S": np.zeros((1, 1, w.dk, w.dv))})
    gs = {n: g[n][:, :, h:h + 1] for n in ("dq", "dk", "dv", "dbeta", "dlam")}
    gs["dS_in"] = g["dS_in"][:, h:h + 1]
    check(w, gs, ref, names=("dq", "dk", "dv", "dbeta", "dlam", "dS_in"))


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
def test_backward_full_size_sampled_heads(F, variant):
    """8 x 2048 x 12 heads of d = 64 in one call; three (b, h) heads are
    recomputed by the oracle one by one (heads are independent)."""
    w = wl(variant, T=2048, B=8, H=12, seed=801)
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 9, device="cuda")
    g = F.backward(params_for(F, w), x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"],
                   c["dS_final"])
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dbeta", "dlam"):
        assert torch.isfinite(g[n].float()).all(), n
    xn = to_np(x)
    cn = to_np(c)
    for b, h in [(0, 0), (3, 7), (7, 11)]:
        sl = lambda a: a[b:b + 1, :, h:h + 1]
        ref = oracle.recurrent_vjp(sl(xn["q"]), sl(xn["k"]), sl(xn["v"]), sl(xn["beta"]),
                                   sl(xn["lam"]), w.variant, sl(cn["dO"]),
                                   cn["dS_final"][b:b + 1, h:h + 1], w.eps, w.eps_gamma)
        gs = {n: g[n][b:b + 1, :, h:h + 1] for n in ("dq", "dk", "dv", "dbeta", "dlam")}
        check(w, gs, ref)
