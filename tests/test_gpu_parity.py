"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle on the
same seeded inputs.  Tolerances: max|o_gpu - o_ref| / max|o_ref| <= 2e-2 for
bf16 inputs (fp32 accumulation) and <= 1e-4 for fp32 inputs, the final
state S to the same bounds."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from helpers import TOL, oracle_full, params_for, rel_err, to_np
from workloads import (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, LM_F1,
                       TINY_F1, Workload, make_carry, make_inputs)

pytestmark = pytest.mark.gpu

ALL = [FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A]


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def run_chunk(F, w, x, carry_in=None, impl=None, T=None):
    p = params_for(F, w, T=T, impl=impl)
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry_in)
    torch.cuda.synchronize()
    return o, co


def medium(variant, dtype="bf16", d=64, T=200, B=2, H=3, chunk=64, W=4, seed=21):
    return Workload(f"medium_v{variant}", variant, B, T, H, d, d, chunk=chunk,
                    window=W if variant in (FALCON_3, FALCON_3A) else 1, dtype=dtype,
                    seed=seed + variant)


def check(w, o, co, o_ref, c_ref, what=""):
    tol = TOL[w.dtype]
    e_o = rel_err(o.float().cpu().numpy(), o_ref)
    e_s = rel_err(co["S"].cpu().numpy(), c_ref["S"])
    assert e_o <= tol and e_s <= tol, f"{what} o {e_o:.3e} S {e_s:.3e} (tol {tol})"
    return e_o, e_s


# ------------------------------------------------------------ chunk forward
@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_chunk_generic_matches_oracle(F, variant, dtype):
    w = medium(variant, dtype)
    x = make_inputs(w, device="cuda")
    o, co = run_chunk(F, w, x, impl=F.FALCON_IMPL_GENERIC)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref, f"variant {variant} {dtype}")
    assert torch.equal(co["k_prev"].cpu(), x["k"][:, -1].cpu())
    assert torch.all(co["pos"].cpu() == w.T)


@pytest.mark.parametrize("variant", ALL)
def test_chunk_auto_matches_oracle(F, variant):
    """The default dispatch (tensor-core path where it applies)."""
    w = medium(variant, "bf16", T=333)
    x = make_inputs(w, device="cuda")
    o, co = run_chunk(F, w, x)
    o_ref, c_ref = oracle_full(w, x)
    check(w, o, co, o_ref, c_ref, f"auto variant {variant}")


@pytest.mark.parametrize("d", [16, 32, 128])
@pytest.mark.parametrize("variant", [FALCON_1, FALCON_2, FALCON_3])
def test_chunk_head_dims(F, variant, d):
    w = medium(variant, "bf16", d=d, T=150, B=1, H=2)
    x = make_inputs(w, device="cuda")
    o, co = run_chunk(F, w, x)
    check(w, o, co, *oracle_full(w, x), what=f"d={d}")


@pytest.mark.parametrize("chunk", [16, 32])
def test_chunk_sizes(F, chunk):
    w = medium(FALCON_1, "f32", chunk=chunk, T=77)
    x = make_inputs(w, device="cuda")
    o, co = run_chunk(F, w, x)
    check(w, o, co, *oracle_full(w, x), what=f"chunk={chunk}")


def test_tiny_reference_case_all_forms(F):
    """1x64x1, d=16, fp32, chunk 16: chunked, masked-parallel and recurrent
    GPU forms all match the oracle to 1e-4."""
    w = TINY_F1
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    o, co = run_chunk(F, w, x)
    check(w, o, co, o_ref, c_ref, "chunked")
    p = params_for(F, w)
    o_m, S_m = F.masked_parallel(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    assert rel_err(o_m.cpu().numpy(), o_ref) <= 1e-4
    assert rel_err(S_m.cpu().numpy(), c_ref["S"]) <= 1e-4
    carry = F.empty_carry(p)
    carry["S"].zero_(); carry["k_prev"].zero_(); carry["pos"].zero_()
    p1 = params_for(F, w, T=1)
    outs = []
    for t in range(w.T):
        o_t = torch.empty((1, 1, 1, w.dv), dtype=x["q"].dtype, device="cuda")
        F.falcon_recurrent_step(p1, x["q"][:, t:t + 1].contiguous(), x["k"][:, t:t + 1].contiguous(),
                                x["v"][:, t:t + 1].contiguous(), x["beta"][:, t:t + 1].contiguous(),
                                x["lam"][:, t:t + 1].contiguous(), carry, o_t)
        outs.append(o_t)
    torch.cuda.synchronize()
    o_r = torch.cat(outs, 1).cpu().numpy()
    assert rel_err(o_r, o_ref) <= 1e-4
    assert rel_err(carry["S"].cpu().numpy(), c_ref["S"]) <= 1e-4


# ------------------------------------------------------------ carry
@pytest.mark.parametrize("variant", ALL)
def test_chunk_carry_round_trip(F, variant):
    """chunk(T1) then chunk(T2) from its carry == oracle over T1 + T2, and the
    carry equals the oracle's (ring and keys bit-exact)."""
    w = medium(variant, "bf16", T=230)
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    T1 = 97
    xa = {k: v[:, :T1].contiguous() for k, v in x.items()}
    xb = {k: v[:, T1:].contiguous() for k, v in x.items()}
    oa, ca = run_chunk(F, w, xa, T=T1)
    ob, cb = run_chunk(F, w, xb, carry_in=ca, T=w.T - T1)
    o = torch.cat([oa, ob], 1)
    check(w, o, cb, o_ref, c_ref, "round trip")
    assert np.array_equal(cb["k_prev"].cpu().double().numpy(), c_ref["k_prev"])
    assert np.array_equal(cb["pos"].cpu().numpy(), c_ref["pos"])
    if "win_x" in c_ref:
        assert np.array_equal(cb["win_x"].cpu().double().numpy(), c_ref["win_x"])
        assert np.array_equal(cb["win_v"].cpu().double().numpy(), c_ref["win_v"])


@pytest.mark.parametrize("variant", ALL)
def test_chunk_from_synthetic_carry(F, variant):
    w = medium(variant, "f32", T=90, d=32)
    x = make_inputs(w, device="cuda")
    carry = make_carry(w, 99, torch.tensor([[0, 1, 5], [2, 40, 3]]), device="cuda")
    o, co = run_chunk(F, w, x, carry_in=carry)
    o_ref, c_ref = oracle_full(w, x, carry)
    check(w, o, co, o_ref, c_ref, "synthetic carry")


@pytest.mark.parametrize("variant", ALL)
def test_chunk_then_recurrent_step(F, variant):
    """chunk(T) then one recurrent step == oracle over T + 1."""
    w = medium(variant, "bf16", T=131)
    x = make_inputs(w, device="cuda")
    o_ref, c_ref = oracle_full(w, x)
    T0 = w.T - 1
    xa = {k: v[:, :T0].contiguous() for k, v in x.items()}
    oa, ca = run_chunk(F, w, xa, T=T0)
    p1 = params_for(F, w, T=1)
    o1 = torch.empty((w.B, 1, w.H, w.dv), dtype=x["q"].dtype, device="cuda")
    F.falcon_recurrent_step(p1, *(x[n][:, T0:].contiguous() for n in ("q", "k", "v", "beta", "lam")),
                            ca, o1)
    torch.cuda.synchronize()
    o = torch.cat([oa, o1], 1)
    check(w, o, ca, o_ref, c_ref, "chunk + step")
    assert np.array_equal(ca["pos"].cpu().numpy(), c_ref["pos"])
    if "win_x" in c_ref:
        assert np.array_equal(ca["win_x"].cpu().double().numpy(), c_ref["win_x"])


# ------------------------------------------------------------ recurrent step
@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_recurrent_step_decode(F, variant, dtype):
    from workloads import make_decode_inputs
    x, carry, w = make_decode_inputs(variant, window=8, B=16, H=12, d=64, dtype=dtype)
    x = {k: v.cuda() for k, v in x.items()}
    carry = {k: v.cuda() for k, v in carry.items()}
    cin = {k: v.clone() for k, v in carry.items()}
    o_ref, c_ref = oracle_full(w, x, cin)
    p = params_for(F, w, T=1)
    o = torch.empty((w.B, 1, w.H, w.dv), dtype=x["q"].dtype, device="cuda")
    F.falcon_recurrent_step(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry, o)
    torch.cuda.synchronize()
    check(w, o, carry, o_ref, c_ref, "decode")
    for key in c_ref:
        if key != "S":
            assert np.array_equal(carry[key].cpu().double().numpy() if key != "pos" else
                                  carry[key].cpu().numpy(), c_ref[key]), key


@pytest.mark.parametrize("variant", [FALCON_1, FALCON_3, FALCON_3A])
def test_recurrent_step_full_size(F, variant):
    """256 x 12 heads, d = 64 (the decode workload the benchmark times): more
    (b, h) items than the window variants' persistent kernel has CTAs, so its
    CTAs walk several items through the double-buffered state; three
    consecutive steps, every head against the oracle."""
    from workloads import make_decode_inputs
    x, carry, w = make_decode_inputs(variant, window=8, B=256, H=12, d=64, seed=17)
    carry = {k: v.cuda() for k, v in carry.items()}
    cref = {k: v.clone().cpu() for k, v in carry.items()}
    p = params_for(F, w, T=1)
    for step in range(3):
        xs, _, _ = make_decode_inputs(variant, window=8, B=256, H=12, d=64, seed=100 + step)
        xs = {k: v.cuda() for k, v in xs.items()}
        o_ref, c_next = oracle_full(w, xs, {k: v.clone() for k, v in cref.items()})
        o = torch.empty((w.B, 1, w.H, w.dv), dtype=xs["q"].dtype, device="cuda")
        F.falcon_recurrent_step(p, xs["q"], xs["k"], xs["v"], xs["beta"], xs["lam"], carry, o)
        torch.cuda.synchronize()
        check(w, o, carry, o_ref, c_next, "decode")
        cref = {k: torch.from_numpy(np.asarray(c)) for k, c in c_next.items()}  # the oracle's own carry, fp64


@pytest.mark.parametrize("d", [16, 32, 128])
def test_recurrent_step_dims(F, d):
    from workloads import make_decode_inputs
    x, carry, w = make_decode_inputs(FALCON_3, window=3, B=4, H=2, d=d, pos=1)
    x = {k: v.cuda() for k, v in x.items()}
    carry = {k: v.cuda() for k, v in carry.items()}
    o_ref, c_ref = oracle_full(w, x, {k: v.clone() for k, v in carry.items()})
    p = params_for(F, w, T=1)
    o = torch.empty((w.B, 1, w.H, w.dv), dtype=x["q"].dtype, device="cuda")
    F.falcon_recurrent_step(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], carry, o)
    torch.cuda.synchronize()
    check(w, o, carry, o_ref, c_ref, f"decode d={d}")


# ------------------------------------------------------------ masked parallel
@pytest.mark.parametrize("variant", ALL)
def test_masked_parallel_ref(F, variant):
    w = medium(variant, "f32", T=96, d=32, W=3)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    o, S = F.masked_parallel(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    o_ref, S_ref = oracle.masked_parallel(*(to_np(x)[n] for n in ("q", "k", "v", "beta", "lam")),
                                          w.variant, w.window)
    assert rel_err(o.cpu().numpy(), o_ref) <= 1e-4
    assert rel_err(S.cpu().numpy(), S_ref) <= 1e-4


# ------------------------------------------------------------ edge cases
@pytest.mark.parametrize("T", [1, 2, 17, 64, 65])
def test_short_sequences(F, T):
    for variant in (FALCON_1, FALCON_3):
        w = medium(variant, "bf16", T=T, B=1, H=2)
        x = make_inputs(w, device="cuda")
        o, co = run_chunk(F, w, x)
        o_ref, c_ref = oracle_full(w, x)
        if T == 1:  # a single fresh token writes nothing: o = 0, S = 0
            assert torch.count_nonzero(o) == 0 and torch.count_nonzero(co["S"]) == 0
        else:
            check(w, o, co, o_ref, c_ref, f"T={T}")


def test_empty_sequence_passes_carry_through(F):
    w = medium(FALCON_3, "bf16", T=5, W=4)
    carry = make_carry(w, 5, 9, device="cuda")
    p = params_for(F, w, T=0)
    co = F.empty_carry(p)
    o = torch.empty((w.B, 0, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    F.falcon_chunk_fwd(p, None, None, None, None, None, carry, o, co)
    torch.cuda.synchronize()
    for key in carry:
        assert torch.equal(co[key], carry[key]), key


def test_forced_zero_decay_clamp(F):
    w = medium(FALCON_1, "bf16", T=400, d=128, B=1, H=2).with_(force_zero_gamma=0.05,
                                                             gamma_mu=4.0, gamma_sd=0.5)
    x = make_inputs(w, device="cuda")
    assert (x["lam"] == 1.0).any()
    o, co = run_chunk(F, w, x)
    assert torch.isfinite(o.float()).all() and torch.isfinite(co["S"]).all()
    check(w, o, co, *oracle_full(w, x), what="clamp")


@pytest.mark.parametrize("beta_val", [1.0, 1e-4])
def test_extreme_steps(F, beta_val):
    w = medium(FALCON_1, "f32", T=150)
    x = make_inputs(w, device="cuda")
    x["beta"].fill_(beta_val)
    o, co = run_chunk(F, w, x)
    check(w, o, co, *oracle_full(w, x), what=f"beta={beta_val}")


def test_zero_keys(F):
    """All-zero keys: every pair has zero energy and the state only decays."""
    w = medium(FALCON_1, "f32", T=70)
    x = make_inputs(w, device="cuda")
    x["k"].zero_()
    o, co = run_chunk(F, w, x)
    assert torch.count_nonzero(o) == 0 and torch.count_nonzero(co["S"]) == 0


# ------------------------------------------------------------ error paths
def test_error_codes(F):
    w = medium(FALCON_1, "bf16", T=10)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    o = torch.empty((w.B, w.T, w.H, w.dv), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd(F.Params(**{**p.__dict__, "dk": 48}), x["q"], x["k"], x["v"],
                           x["beta"], x["lam"], None, o, None)
    assert e.value.code == -2
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd(p, None, x["k"], x["v"], x["beta"], x["lam"], None, o, None)
    assert e.value.code == -1
    c = F.empty_carry(p)
    with pytest.raises(F.FalconError) as e:  # carry_in and carry_out overlap
        F.falcon_chunk_fwd(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], c, o, c)
    assert e.value.code == -1
