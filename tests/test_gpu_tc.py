"""Tensor-core chunk path (tcgen05 / TMEM / TMA): parity with the oracle when
forced, agreement with the portable path, and a white-box check of the
per-chunk WY stage and what it leaves in the workspace, with T = (I + A)^{-1}:
the bf16 images of W = T diag(eta Gamma) X and U = T diag(eta) V (d / 64
slabs of 64 columns each, d = 64 and 128) and the decay gates of the
sequential kernel."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import TOL, oracle_full, params_for, rel_err
from workloads import FALCON_1, FALCON_1A, LM_F1, Workload, make_carry, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def w_tc(variant, d=64, T=300, B=2, H=2, seed=31):
    return Workload(f"tc_v{variant}_d{d}", variant, B, T, H, d, d, chunk=64, seed=seed + variant)


def decode_T(img: np.ndarray) -> np.ndarray:
    """bf16 image of a 64x64 K-major tile with the 128-byte swizzle -> matrix."""
    raw = img.view(np.uint16).reshape(-1)
    out = np.zeros((64, 64), dtype=np.float32)
    for R in range(64):
        for j in range(8):
            base = (R * 128 + 16 * (j ^ (R & 7))) // 2
            vals = raw[base:base + 8].astype(np.uint32) << 16
            out[R, 8 * j:8 * j + 8] = vals.view(np.float32)
    return out


@pytest.mark.parametrize("d", [64, 128])
def test_wy_stage_workspace(F, d):
    w = w_tc(FALCON_1, d=d, T=150, B=1, H=2)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    n = F.falcon_workspace_size(p)
    ws = F.alloc_workspace(n)
    ws.zero_()
    F.falcon_chunk_fwd(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, None, ws, n)
    torch.cuda.synchronize()
    NC = (w.T + 63) // 64
    wsn = ws.cpu().numpy()
    assert int(wsn[:4].view(np.uint32)[0]) == 0, "status word set"
    t_off = 256
    img_bytes = 2 * d * 128  # W slabs | U slabs
    g_off = t_off + w.B * w.H * NC * img_bytes
    k = x["k"].float().cpu().numpy().astype(np.float64)
    vv = x["v"].float().cpu().numpy().astype(np.float64)
    lam = x["lam"].cpu().numpy().astype(np.float64)
    beta = x["beta"].cpu().numpy().astype(np.float64)
    for bh in range(w.B * w.H):
        b, h = divmod(bh, w.H)
        for c in range(NC):
            rows = np.arange(c * 64, c * 64 + 64)
            X = np.zeros((64, d))
            for r, t in enumerate(rows):
                if 1 <= t < w.T:
                    X[r] = k[b, t - 1, h]
            ok = rows < w.T
            ell = np.where(ok, np.log(np.clip(1 - lam[b, np.minimum(rows, w.T - 1), h], 1e-3, 1)), 0)
            g = np.cumsum(ell)
            G = X @ X.T
            eta = np.where(ok & (rows >= 1), beta[b, np.minimum(rows, w.T - 1), h] / (1e-6 + np.diag(G)), 0)
            A = eta[:, None] * np.exp(np.minimum(g[:, None] - g[None, :], 0)) * G * np.tril(np.ones((64, 64)), -1)
            Tref = np.linalg.inv(np.eye(64) + A)
            ci = bh * NC + c
            img = wsn[t_off + ci * img_bytes: t_off + (ci + 1) * img_bytes]
            Tw_ref = Tref * (eta * np.exp(g))[None, :]
            Tu_ref = Tref * eta[None, :]
            V = np.zeros((64, d))
            V[ok] = vv[b, rows[ok], h]
            slabs = range(d // 64)
            got_W = np.hstack([decode_T(img[8192 * sl:8192 * (sl + 1)]) for sl in slabs])
            got_U = np.hstack([decode_T(img[d * 128 + 8192 * sl:d * 128 + 8192 * (sl + 1)]) for sl in slabs])
            for got, ref in ((got_W, Tw_ref @ X), (got_U, Tu_ref @ V)):
                assert np.abs(got - ref).max() <= 2e-2 * max(np.abs(ref).max(), 1e-30), (bh, c)
            # Gamma, exp(g_last - g), g, exp(g - g at the start of the 16-row block)
            gates = wsn[g_off + ci * 1024: g_off + (ci + 1) * 1024].view(np.float32)
            assert np.allclose(gates[:64], np.exp(g), rtol=1e-4, atol=1e-6), (bh, c)
            assert np.allclose(gates[64:128], np.exp(g[-1] - g), rtol=1e-4, atol=1e-6), (bh, c)
            assert np.allclose(gates[128:192], g, rtol=1e-4, atol=1e-5), (bh, c)
            assert np.allclose(gates[192:256], np.exp(g - g[np.arange(64) & ~15]), rtol=1e-4,
                               atol=1e-6), (bh, c)


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
@pytest.mark.parametrize("d", [64, 128])
def test_tc_forced_matches_oracle(F, variant, d):
    w = w_tc(variant, d=d)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x)
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= TOL["bf16"] and e_s <= TOL["bf16"], (e_o, e_s)
    assert torch.equal(co["k_prev"].cpu(), x["k"][:, -1].cpu())
    assert torch.all(co["pos"].cpu() == w.T)


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
def test_tc_with_carry(F, variant):
    w = w_tc(variant, T=200, B=2, H=3)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 77, torch.tensor([[0, 3, 64], [1, 2, 500]]), device="cuda")
    p = params_for(F, w, impl=F.FALCON_IMPL_TC)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry)
    torch.cuda.synchronize()
    o_ref, c_ref = oracle_full(w, x, carry)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]
    assert rel_err(co["S"].cpu().numpy(), c_ref["S"]) <= TOL["bf16"]
    assert np.array_equal(co["pos"].cpu().numpy(), c_ref["pos"])


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
def test_tc_agrees_with_generic(F, variant):
    w = w_tc(variant, T=513, B=1, H=4)
    x = make_inputs(w, device="cuda")
    outs = {}
    for impl in (F.FALCON_IMPL_TC, F.FALCON_IMPL_GENERIC):
        p = params_for(F, w, impl=impl)
        outs[impl] = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    (o1, c1), (o2, c2) = outs[F.FALCON_IMPL_TC], outs[F.FALCON_IMPL_GENERIC]
    assert rel_err(o1.float().cpu().numpy(), o2.float().cpu().numpy()) <= TOL["bf16"]
    assert rel_err(c1["S"].cpu().numpy(), c2["S"].cpu().numpy()) <= TOL["bf16"]


def test_tc_full_size_sampled_heads(F):
    """Falcon-1, 8 x 2048 x 12 heads, d = 64, bf16, in the launch
    configuration the benchmark times; sampled heads against the oracle."""
    import oracle
    w = LM_F1
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    heads = [(0, 0), (3, 7), (7, 11)]
    xn = {k: v.cpu().double().numpy() for k, v in x.items()}
    o_ref, S_ref = oracle.recurrent_heads(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"],
                                          w.variant, heads)
    for i, (b, h) in enumerate(heads):
        assert rel_err(o[b, :, h].float().cpu().numpy(), o_ref[i]) <= TOL["bf16"]
        assert rel_err(co["S"][b, h].cpu().numpy(), S_ref[i]) <= TOL["bf16"]
    assert torch.isfinite(o.float()).all()


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_1A])
def test_tc_long_clamped_runs(F, variant):
    """Runs of clamped decay (lambda = 1, gamma = eps_gamma) long enough that
    the in-block decay ratios underflow fp32: the kernels must fall back to
    exact per-element decays there."""
    w = w_tc(variant, T=300, B=1, H=2, seed=7)
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
