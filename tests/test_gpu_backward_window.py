"""Backward pass of the window variants (Falcon-3/3A) and of every variant at
d = 128 (falcon_backward_carry through the C ABI) against the backward
oracle (torch fp64 autodiff of the recurrence with its window of pairs):
every gradient element by element, windows 2..64, both pairings, bf16 and
fp32, d = 32, 64 and 128, the carried state, key and window ring (gradients
of all three), clamped decays, the empty and one-step sequences, block
boundaries (64 steps), and, at 4 x 8192 x 12 d64 W = 8 in one call, sampled
heads computed one by one."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import params_for, rel_err, to_np
from workloads import (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, WINDOW_F3, Workload,
                       make_carry, make_cotangents, make_inputs)

pytestmark = pytest.mark.gpu

# as for the one-pair backward: dq, dk, dv and the ring gradients are stored
# in the dtype; dbeta, dlam and dS_in are fp32 results
TOL_D = {"bf16": 2e-2, "f32": 1e-3}
TOL_F32 = {"bf16": 2e-3, "f32": 1e-3}
IN_DTYPE = ("dq", "dk", "dv", "dk_prev", "dwin_x", "dwin_v")
ALL = ("dq", "dk", "dv", "dbeta", "dlam", "dS_in", "dk_prev")


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def wl(variant, W, d=64, T=150, B=2, H=3, dtype="bf16", pairing="prefix", seed=901, **kw):
    return Workload(f"bwdw_v{variant}_w{W}_d{d}", variant, B, T, H, d, d, chunk=64, dtype=dtype,
                    window=W, seed=seed + variant + 7 * W, pairing=pairing, **kw)


def run_both(F, w, carry=None, with_dS=True, cot_seed=5):
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, cot_seed, device="cuda", with_dS=with_dS)
    p = params_for(F, w)
    g = F.backward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"], c["dS_final"], carry)
    torch.cuda.synchronize()
    xn = to_np(x)
    cn = to_np({k: v for k, v in c.items() if v is not None})
    ref = oracle.recurrent_vjp(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"], w.variant,
                               cn["dO"], cn.get("dS_final"), w.eps, w.eps_gamma,
                               carry=to_np(carry), pairing=w.pairing, window=w.window)
    return g, ref


def check(w, g, ref, names=("dq", "dk", "dv", "dbeta", "dlam")):
    errs = {}
    for n in names:
        tol = TOL_D[w.dtype] if n in IN_DTYPE else TOL_F32[w.dtype]
        e = rel_err(g[n].double().cpu().numpy(), ref[n])
        errs[n] = e
        assert e <= tol, (n, e, errs)
    return errs


@pytest.mark.parametrize("variant", [FALCON_3, FALCON_3A])
@pytest.mark.parametrize("W", [2, 3, 8])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_window_backward_matches_oracle(F, variant, W, pairing):
    w = wl(variant, W, pairing=pairing)
    assert F.falcon_backward_workspace_size(params_for(F, w)) > 0
    g, ref = run_both(F, w)
    check(w, g, ref)
    assert torch.isfinite(g["dS_in"]).all()


@pytest.mark.parametrize("variant", [FALCON_3, FALCON_3A])
def test_window_backward_f32(F, variant):
    w = wl(variant, 5, dtype="f32", T=130, seed=913)
    carry = make_carry(w, seed=21, pos=torch.tensor([[0, 2, 9], [1, 40, 3]]), device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=ALL + ("dwin_x", "dwin_v"))


@pytest.mark.parametrize("variant", [FALCON_3, FALCON_3A])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
@pytest.mark.parametrize("W", [4, 8])
def test_window_backward_with_carried_ring(F, variant, pairing, W):
    """Carried state, key, ring and positions (0, 1, a few and many tokens
    consumed): the ring slots of pairs that exist get their gradients, the
    others zero."""
    w = wl(variant, W, T=140, pairing=pairing, seed=921)
    pos = torch.tensor([[0, 1, 3], [300, 2, 57]], dtype=torch.int64)
    carry = make_carry(w, seed=22, pos=pos, device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=ALL + ("dwin_x", "dwin_v"))


@pytest.mark.parametrize("d", [32, 128])
@pytest.mark.parametrize("variant", [FALCON_3, FALCON_3A])
def test_window_backward_head_dims(F, d, variant):
    w = wl(variant, 4, d=d, T=100, seed=931)
    carry = make_carry(w, seed=23, pos=torch.tensor([[0, 5, 2], [9, 1, 70]]), device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=ALL + ("dwin_x", "dwin_v"))


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A, FALCON_2, FALCON_2A])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_backward_d128_one_pair(F, variant, pairing):
    w = wl(variant, 1, d=128, T=150, pairing=pairing, seed=941)
    carry = make_carry(w, seed=24, pos=torch.tensor([[0, 1, 40], [2, 0, 300]]), device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=ALL)


@pytest.mark.parametrize("W,d", [(64, 64), (34, 128), (17, 32)])
def test_window_backward_wide_windows(F, W, d):
    """The widest windows the kernel takes (two or more reduction groups of
    eight pairs, and a group that is not full)."""
    w = wl(FALCON_3, W, d=d, T=90, B=1, H=2, seed=951)
    carry = make_carry(w, seed=25, pos=torch.tensor([[3, 200]]), device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=ALL + ("dwin_x", "dwin_v"))


@pytest.mark.parametrize("T", [1, 2, 7, 63, 64, 65, 129])
def test_window_backward_block_edges(F, T):
    w = wl(FALCON_3, 8, T=T, B=1, H=2, seed=961)
    carry = make_carry(w, seed=26, pos=torch.tensor([[4, 100]]), device="cuda")
    g, ref = run_both(F, w, carry=carry)
    check(w, g, ref, names=ALL + ("dwin_x", "dwin_v"))


def test_window_backward_empty_sequence(F):
    w = wl(FALCON_3, 6, T=0, B=2, H=2)
    carry = make_carry(w, seed=27, pos=9, device="cuda")
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 3, device="cuda")
    g = F.backward(params_for(F, w), x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"],
                   c["dS_final"], carry)
    torch.cuda.synchronize()
    assert torch.equal(g["dS_in"], c["dS_final"])
    for n in ("dk_prev", "dwin_x", "dwin_v"):
        assert float(g[n].float().abs().max()) == 0.0, n


@pytest.mark.parametrize("variant", [FALCON_3, FALCON_3A])
def test_window_backward_clamped_decay(F, variant):
    w = wl(variant, 8, T=160, force_zero_gamma=0.2, gamma_mu=-1.0, gamma_sd=3.0, seed=971)
    g, ref = run_both(F, w)
    check(w, g, ref)
    lam = make_inputs(w)["lam"]
    clamped = (1.0 - lam) < w.eps_gamma
    assert clamped.any()
    assert float(g["dlam"].cpu()[clamped].abs().max()) == 0.0


def test_window_backward_without_ring_outputs(F):
    """falcon_backward (no ring gradients) returns the same gradients as
    falcon_backward_carry."""
    w = wl(FALCON_3, 4, T=70, B=1, H=2, seed=981)
    carry = make_carry(w, seed=28, pos=torch.tensor([[6, 1]]), device="cuda")
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 4, device="cuda")
    p = params_for(F, w)
    g = F.backward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"], c["dS_final"], carry)
    h = {n: torch.empty_like(g[n]) for n in ("dq", "dk", "dv", "dbeta", "dlam", "dS_in", "dk_prev")}
    n_ws = F.falcon_backward_workspace_size(p)
    ws = F.alloc_workspace(n_ws)
    F.falcon_backward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry, c["dO"], c["dS_final"],
                      h["dq"], h["dk"], h["dv"], h["dbeta"], h["dlam"], h["dS_in"], h["dk_prev"], ws, n_ws)
    torch.cuda.synchronize()
    for n, t in h.items():
        assert torch.equal(t, g[n]), n


def test_window_backward_full_size_sampled_heads(F):
    """Falcon-3, 4 x 8192 x 12 heads, d = 64, W = 8 in one call; two (b, h)
    heads are recomputed by the oracle one by one (heads are independent)."""
    w = WINDOW_F3
    x = make_inputs(w, device="cuda")
    c = make_cotangents(w, 9, device="cuda")
    g = F.backward(params_for(F, w), x["q"], x["k"], x["v"], x["beta"], x["lam"], c["dO"],
                   c["dS_final"])
    torch.cuda.synchronize()
    for n in ("dq", "dk", "dv", "dbeta", "dlam", "dS_in"):
        assert torch.isfinite(g[n].float()).all(), n
    xn = to_np(x)
    cn = to_np(c)
    for b, h in [(0, 0), (3, 11)]:
        sl = lambda a: a[b:b + 1, :, h:h + 1]
        ref = oracle.recurrent_vjp(sl(xn["q"]), sl(xn["k"]), sl(xn["v"]), sl(xn["beta"]),
                                   sl(xn["lam"]), w.variant, sl(cn["dO"]),
                                   cn["dS_final"][b:b + 1, h:h + 1], w.eps, w.eps_gamma, window=w.window,
                                   carry={"S": np.zeros((1, 1, w.dk, w.dv))})  # a zero state: fresh
        gs = {n: g[n][b:b + 1, :, h:h + 1] for n in ("dq", "dk", "dv", "dbeta", "dlam")}
        gs["dS_in"] = g["dS_in"][b:b + 1, h:h + 1]
        check(w, gs, ref, names=("dq", "dk", "dv", "dbeta", "dlam", "dS_in"))
