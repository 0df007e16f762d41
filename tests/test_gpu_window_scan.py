"""Falcon-3 window recurrence (FALCON_IMPL_SCAN) against the oracle through
the C ABI: windows 2..8, d_k = 32 / 64, bf16 and fp32, several staged blocks
with a ragged tail, carries in and out (window rings bit-exact with the
portable chunk kernel's), fresh and continued sequences with the window not
yet full, same-step pairing, empty and one-step calls, clamped decays, and
sampled heads of the 4 x 8192 x 12, d = 64, W = 8 workload (forced: AUTO
takes the tensor-core path at d = 64 in bf16)."""

from __future__ import annotations

import pytest
import torch

import oracle
from helpers import TOL, oracle_full, params_for, rel_err, to_np
from workloads import FALCON_1, FALCON_3, WINDOW_F3, Workload, make_carry, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def wl(W=8, d=64, T=200, B=2, H=2, dtype="bf16", pairing="prefix", seed=901, **kw):
    return Workload(f"scan_w{W}_d{d}", FALCON_3, B, T, H, d, d, window=W, dtype=dtype, seed=seed + W,
                    pairing=pairing, **kw)


def run(F, w, x, carry=None, impl=None, T=None):
    p = params_for(F, w, T=T, impl=F.FALCON_IMPL_SCAN if impl is None else impl)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    return o, co


def check(w, o, co, o_ref, c_ref):
    tol = TOL[w.dtype]
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= tol and e_s <= tol, (e_o, e_s, tol)


@pytest.mark.parametrize("W", [2, 3, 5, 8])
@pytest.mark.parametrize("d", [32, 64])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_scan_matches_oracle(F, W, d, dtype):
    w = wl(W=W, d=d, dtype=dtype)
    auto = F.falcon_chunk_fwd_plan(params_for(F, w))[0]  # d = 64 bf16 runs on the tensor cores
    assert auto == (F.FALCON_IMPL_TC if (d == 64 and dtype == "bf16") else F.FALCON_IMPL_SCAN)
    x = make_inputs(w, device="cuda")
    o, co = run(F, w, x)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref)


@pytest.mark.parametrize("W", [3, 8])
@pytest.mark.parametrize("pos", [0, 1, 2, 5, 100])
def test_scan_from_carry(F, W, pos):
    w = wl(W=W, T=150, seed=911)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, seed=31 + pos, pos=pos, device="cuda")
    o, co = run(F, w, x, carry)
    o_ref, c_ref = oracle_full(w, x, carry)
    check(w, o, co, o_ref, c_ref)
    _, co_g = run(F, w, x, carry, impl=F.FALCON_IMPL_GENERIC)
    for n in ("k_prev", "win_x", "win_v", "pos"):
        assert torch.equal(co[n], co_g[n]), n


@pytest.mark.parametrize("W", [4, 8])
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_scan_carry_round_trip(F, W, pairing):
    w = wl(W=W, T=230, pairing=pairing, seed=921)
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    T1 = 97
    x1 = {k: v[:, :T1].contiguous() for k, v in x.items()}
    x2 = {k: v[:, T1:].contiguous() for k, v in x.items()}
    o1, c1 = run(F, w, x1, T=T1)
    o2, c2 = run(F, w, x2, c1, T=w.T - T1)
    o = torch.cat([o1, o2], dim=1)
    check(w, o, c2, o_ref, c_ref)
    assert int(c2["pos"].min()) == w.T


@pytest.mark.parametrize("T", [0, 1, 2, 62, 63, 64, 127])
def test_scan_short_and_block_edges(F, T):
    w = wl(W=8, T=T, B=1, H=3, seed=931)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, seed=41, pos=3, device="cuda")
    o, co = run(F, w, x, carry)
    if T == 0:  # nothing to compute: the carry passes through
        for n in ("S", "k_prev", "win_x", "win_v", "pos"):
            assert torch.equal(co[n], carry[n]), n
        return
    o_ref, c_ref = oracle_full(w, x, carry)
    check(w, o, co, o_ref, c_ref)


def test_scan_clamped_decay(F):
    w = wl(W=8, T=300, force_zero_gamma=0.05, gamma_mu=4.0, gamma_sd=0.5, seed=941)
    x = make_inputs(w, device="cuda")
    o, co = run(F, w, x)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref)


def test_scan_coverage(F):
    w = wl(W=8)
    with pytest.raises(F.FalconError) as e:  # forced on a shape it does not cover
        F.falcon_chunk_fwd_plan(params_for(F, w.with_(window=9), impl=F.FALCON_IMPL_SCAN))
    assert e.value.code == -2
    w9 = w.with_(window=9, T=40)
    with pytest.raises(F.FalconError) as e:
        run(F, w9, make_inputs(w9, device="cuda"))
    assert e.value.code == -2
    p = params_for(F, w.with_(window=9), impl=F.FALCON_IMPL_AUTO)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    p = params_for(F, w.with_(window=10), impl=F.FALCON_IMPL_AUTO)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_GENERIC
    p = params_for(F, w.with_(variant=FALCON_1, window=1), impl=F.FALCON_IMPL_SCAN)
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd_plan(p)
    assert e.value.code == -2
    p = params_for(F, w.with_(dk=16, dv=16), impl=F.FALCON_IMPL_AUTO)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_GENERIC


def test_scan_full_size_sampled_heads(F):
    """Falcon-3, 4 x 8192 x 12 heads, d = 64, W = 8 in one call (the launch
    the benchmark times); three heads recomputed by the oracle's recurrence."""
    w = WINDOW_F3
    p = params_for(F, w, impl=F.FALCON_IMPL_SCAN)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_SCAN
    x = make_inputs(w, device="cuda")
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all()
    xn = to_np(x)
    for b, h in [(0, 0), (2, 5), (3, 11)]:
        sl = {n: a[b:b + 1, :, h:h + 1] for n, a in xn.items()}
        o_ref, c_ref = oracle.recurrent(sl["q"], sl["k"], sl["v"], sl["beta"], sl["lam"], w.variant,
                                        w.window, w.eps, w.eps_gamma)
        e_o = rel_err(o[b:b + 1, :, h:h + 1].float().cpu().numpy(), o_ref)
        e_s = rel_err(co["S"][b:b + 1, h:h + 1].cpu().numpy(), c_ref["S"])
        assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (b, h, e_o, e_s)


def test_scan_misaligned_tensors(F):
    """Rows not on a 16-byte boundary: AUTO takes the portable kernel (same
    result), a forced SCAN is refused."""
    w = wl(W=4, T=90, B=1, H=2, seed=951)
    x = make_inputs(w, device="cuda")
    q2 = torch.empty(x["q"].numel() + 1, dtype=x["q"].dtype, device="cuda")
    q2[1:].copy_(x["q"].reshape(-1))
    xq = dict(x, q=q2[1:].view(x["q"].shape))
    assert xq["q"].data_ptr() % 16 != 0
    o, co = run(F, w, xq, impl=F.FALCON_IMPL_AUTO)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref)
    with pytest.raises(F.FalconError) as e:
        run(F, w, xq)
    assert e.value.code == -1
