"""Prologue (phi = per-token L2 normalisation of q and k, gates from
logits) and packed variable-length sequences, through the C ABI, against
the oracle (prologue applied in fp64, each sequence run on its own): every
variant on its default kernel family, bf16 and fp32, lengths 0 / 1 / block
and chunk edges, per-sequence carries in and out (keys, positions, window
rings bit-exact), the recurrent step with the prologue, and the calls that
must refuse a prologue."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, params_for, rel_err, to_np
from workloads import (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, Workload,
                       make_carry, make_inputs, make_raw_inputs, pack_varlen)

pytestmark = pytest.mark.gpu

ALL = [FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A]
BOTH = 3  # L2NORM_QK | GATE_LOGITS


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def wl(variant, T=150, B=2, H=2, d=64, dtype="bf16", W=4, seed=1001, pairing="prefix"):
    return Workload(f"vl_v{variant}", variant, B, T, H, d, d,
                    window=W if variant in (FALCON_3, FALCON_3A) else 1, dtype=dtype,
                    seed=seed + variant, pairing=pairing)


def oracle_pro(w, x, flags, carry=None):
    xn = to_np(x)
    q, k, b, l = oracle.apply_prologue(xn["q"], xn["k"], xn["beta"], xn["lam"], flags)
    return oracle.recurrent(q, k, xn["v"], b, l, w.variant, w.window, w.eps, w.eps_gamma,
                            carry=to_np(carry), pairing=w.pairing)


def check(w, o, S, o_ref, S_ref):
    tol = TOL[w.dtype]
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(S.cpu().numpy(), S_ref)
    assert e_o <= tol and e_s <= tol, (e_o, e_s, tol)


@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("flags", [1, 2, BOTH])
def test_prologue_dense(F, variant, flags):
    w = wl(variant)
    x = make_raw_inputs(w, device="cuda")
    if not flags & 2:  # gates given directly
        g = make_inputs(w, device="cuda")
        x["beta"], x["lam"] = g["beta"], g["lam"]
    p = params_for(F, w)
    p.prologue = flags
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_pro(w, x, flags)
    check(w, o, co["S"], o_ref, c_ref["S"])
    if flags & 1:  # the carried key is a feature
        assert np.allclose(np.linalg.norm(co["k_prev"].float().cpu().numpy(), axis=-1), 1.0, atol=1e-2)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_prologue_dense_fp32_and_timed_plan(F, dtype):
    """bf16 Falcon-1 at d = 64 takes the prologue inside its two kernels (no
    extra launch); the fp32 path applies it in a gather pass first."""
    w = wl(FALCON_1, dtype=dtype)
    x = make_raw_inputs(w, device="cuda")
    p = params_for(F, w)
    p.prologue = BOTH
    impl, launches = F.falcon_chunk_fwd_plan(p)
    p0 = params_for(F, w)
    assert launches == F.falcon_chunk_fwd_plan(p0)[1] + (0 if dtype == "bf16" else 1)
    assert F.falcon_workspace_size(p) > F.falcon_workspace_size(p0)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_pro(w, x, BOTH)
    check(w, o, co["S"], o_ref, c_ref["S"])


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
@pytest.mark.parametrize("flags", [1, BOTH])
def test_prologue_fused_continuation(F, variant, pairing, flags):
    """The prologue inside the d = 64 tensor-core kernels across two calls:
    the second takes the first's carry (its carried key a feature), and the
    two outputs and the final state match the oracle on the whole sequence."""
    T1, T2 = 100, 150
    w = wl(variant, T=T1 + T2, pairing=pairing)
    x = make_raw_inputs(w, device="cuda")
    if not flags & 2:
        g = make_inputs(w, device="cuda")
        x["beta"], x["lam"] = g["beta"], g["lam"]
    outs, carry = [], None
    for t0, t1 in ((0, T1), (T1, T1 + T2)):
        wp = w.with_(T=t1 - t0)
        p = params_for(F, wp)
        p.prologue = flags
        assert F.falcon_chunk_fwd_plan(p)[1] == F.falcon_chunk_fwd_plan(params_for(F, wp))[1]
        xs = {n: v[:, t0:t1].contiguous() for n, v in x.items()}
        o, carry = F.chunk_forward(p, xs["q"], xs["k"], xs["v"], xs["beta"], xs["lam"], carry)
        outs.append(o)
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_pro(w, x, flags)
    check(w, torch.cat(outs, dim=1), carry["S"], o_ref, c_ref["S"])


def varlen_case(F, w, lengths, flags=0, carries=None, raw=False):
    T = max(max(lengths), 1)
    wfull = w.with_(B=len(lengths), T=T)
    x = make_raw_inputs(wfull, device="cpu") if raw else make_inputs(wfull, device="cpu")
    packed, cu = pack_varlen(x, lengths, device="cuda")
    p = params_for(F, wfull)
    p.prologue = flags
    ci = None
    if carries is not None:
        ci = make_carry(wfull, seed=77, pos=torch.tensor(carries).repeat_interleave(w.H), device="cuda")
    o, co = F.chunk_forward_varlen(p, cu, packed["q"], packed["k"], packed["v"], packed["beta"],
                                   packed["lam"], ci)
    torch.cuda.synchronize()
    pn = to_np(packed)
    q, k, b, l = oracle.apply_prologue(pn["q"], pn["k"], pn["beta"], pn["lam"], flags)
    cin = None
    if ci is not None:
        cn = to_np(ci)
        cin = [{n: a[i:i + 1] for n, a in cn.items()} for i in range(len(lengths))]
    o_ref, cos = oracle.recurrent_varlen(q, k, pn["v"], b, l, cu.cpu().numpy(), w.variant, w.window,
                                         w.eps, w.eps_gamma, carries=cin, pairing=w.pairing)
    return wfull, o, co, o_ref, cos, ci, x, packed, cu


@pytest.mark.parametrize("variant", ALL)
def test_varlen_matches_separate_sequences(F, variant):
    lengths = [200, 0, 1, 63, 64, 65, 130]
    w = wl(variant)
    wfull, o, co, o_ref, cos, _, x, packed, cu = varlen_case(F, w, lengths)
    tol = TOL[w.dtype]
    assert rel_err(o.float().cpu().numpy(), o_ref) <= tol
    for i, L in enumerate(lengths):
        S_ref = np.zeros((1, w.H, w.dk, w.dv)) if cos[i] is None else cos[i]["S"]
        assert rel_err(co["S"][i:i + 1].cpu().numpy(), S_ref) <= tol or np.abs(S_ref).max() == 0, i
        assert int(co["pos"][i].min()) == L
        if L > 0:  # last key, and the ring, bit-exact with a dense call on that sequence alone
            xb = {n: t[i:i + 1, :L].contiguous().cuda() for n, t in x.items()}
            _, cb = F.chunk_forward(params_for(F, w.with_(B=1, T=L), impl=F.FALCON_IMPL_GENERIC),
                                    xb["q"], xb["k"], xb["v"], xb["beta"], xb["lam"])
            torch.cuda.synchronize()
            for n in ("k_prev", "win_x", "win_v"):
                if n in co:
                    assert torch.equal(co[n][i], cb[n][0]), (i, n)


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_2, FALCON_3])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_varlen_with_carries_and_prologue(F, variant, pairing):
    lengths = [97, 3, 0, 64]
    w = wl(variant, pairing=pairing, seed=1101)
    wfull, o, co, o_ref, cos, ci, *_ = varlen_case(F, w, lengths, flags=BOTH, carries=[5, 0, 2, 130],
                                                   raw=True)
    tol = TOL[w.dtype]
    assert rel_err(o.float().cpu().numpy(), o_ref) <= tol
    for i, L in enumerate(lengths):
        if L == 0:  # nothing consumed: the carry passes through
            assert torch.equal(co["S"][i], ci["S"][i]) and torch.equal(co["k_prev"][i], ci["k_prev"][i])
            continue
        assert rel_err(co["S"][i:i + 1].cpu().numpy(), cos[i]["S"]) <= tol, i
        assert np.array_equal(co["pos"][i].cpu().numpy(), cos[i]["pos"][0]), i


def test_varlen_fp32(F):
    w = wl(FALCON_1A, dtype="f32")
    lengths = [40, 1, 77]
    wfull, o, co, o_ref, cos, *_ = varlen_case(F, w, lengths)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL["f32"]


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_2, FALCON_3])
def test_recurrent_step_prologue(F, variant):
    w = wl(variant, T=6, B=3, H=2, seed=1201)
    x = make_raw_inputs(w, device="cuda")
    carry = make_carry(w, seed=9, pos=7, device="cuda")
    o_ref, c_ref = oracle_pro(w, x, BOTH, carry)
    p = params_for(F, w, T=1)
    p.prologue = BOTH
    c = {n: t.clone() for n, t in carry.items()}
    outs = []
    for t in range(w.T):
        xt = {n: a[:, t:t + 1].contiguous() for n, a in x.items()}
        o = torch.empty((w.B, 1, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
        F.falcon_recurrent_step(p, xt["q"], xt["k"], xt["v"], xt["beta"], xt["lam"], c, o)
        outs.append(o)
    torch.cuda.synchronize()
    check(w, torch.cat(outs, dim=1), c["S"], o_ref, c_ref["S"])


def test_prologue_refused_where_not_taken(F):
    w = wl(FALCON_1, T=8, B=1, H=1)
    p = params_for(F, w)
    p.prologue = 4
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd_plan(p)
    assert e.value.code == -1
    p.prologue = 1
    x = make_inputs(w, device="cuda")
    with pytest.raises(F.FalconError) as e:
        F.masked_parallel(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    assert e.value.code == -2
    assert F.falcon_backward_workspace_size(p) == 0
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd_noalloc(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None,
                                   torch.empty_like(x["v"]), None)
    assert e.value.code == -2


def test_prologue_misaligned_rows(F):
    """q off a 16-byte boundary: the gather pass takes its element-wise form."""
    w = wl(FALCON_1, T=70, B=1, H=2, seed=1301)
    x = make_raw_inputs(w, device="cuda")
    q2 = torch.empty(x["q"].numel() + 1, dtype=x["q"].dtype, device="cuda")
    q2[1:].copy_(x["q"].reshape(-1))
    xq = dict(x, q=q2[1:].view(x["q"].shape))
    assert xq["q"].data_ptr() % 16 != 0
    p = params_for(F, w)
    p.prologue = BOTH
    o, co = F.chunk_forward(p, xq["q"], xq["k"], xq["v"], xq["beta"], xq["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_pro(w, x, BOTH)
    check(w, o, co["S"], o_ref, c_ref["S"])


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
def test_varlen_in_place_carry_without_key(F, variant):
    """Packed rows read in place: a sequence that continues (pos > 0) with no
    carried key pairs its first value with a zero key, never with the
    previous sequence's last key, which sits on the row before it."""
    lengths = [70, 5, 131]
    w = wl(variant, seed=1201)
    T = max(lengths)
    wfull = w.with_(B=len(lengths), T=T)
    x = make_inputs(wfull, device="cpu")
    packed, cu = pack_varlen(x, lengths, device="cuda")
    p = params_for(F, wfull)
    ci = make_carry(wfull, seed=78, pos=torch.tensor([3, 9, 1]).repeat_interleave(w.H), device="cuda")
    del ci["k_prev"]
    o, co = F.chunk_forward_varlen(p, cu, packed["q"], packed["k"], packed["v"], packed["beta"],
                                   packed["lam"], ci)
    torch.cuda.synchronize()
    pn = to_np(packed)
    cn = to_np(ci)
    cin = [{n: a[i:i + 1] for n, a in cn.items()} for i in range(len(lengths))]
    o_ref, cos = oracle.recurrent_varlen(pn["q"], pn["k"], pn["v"], pn["beta"], pn["lam"], cu.cpu().numpy(),
                                         w.variant, w.window, w.eps, w.eps_gamma, carries=cin, pairing=w.pairing)
    tol = TOL[w.dtype]
    assert rel_err(o.float().cpu().numpy(), o_ref) <= tol
    for i in range(len(lengths)):
        assert rel_err(co["S"][i:i + 1].cpu().numpy(), cos[i]["S"]) <= tol, i
