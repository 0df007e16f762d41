"""Pins of the backward oracle (oracle/falcon_grad.py).

G1  its torch forward equals the numpy oracle's recurrence (every one-pair
    variant, carries, both pairings), so the function being differentiated
    is the pinned forward
G2  its gradients equal central finite differences of
    L = <o, do> + <S_final, dS_final> for every input, including the carried
    state and key
G3  a clamped decay passes no gradient to lambda, and a step whose pair does
    not exist passes none to beta
"""

import numpy as np
import pytest

import oracle as O

ONE = [O.FALCON_1, O.FALCON_1A, O.FALCON_2, O.FALCON_2A]


def inputs(rng, B, T, H, dk, dv, per_channel):
    q = rng.standard_normal((B, T, H, dk))
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    bshape = (B, T, H, dv) if per_channel else (B, T, H)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(bshape)))
    lam = 1.0 / (1.0 + np.exp(-(rng.standard_normal((B, T, H)) - 2.0)))   # inside (0, 1 - eps_gamma)
    return dict(q=q, k=k, v=v, beta=beta, lam=lam)


def carry_for(rng, B, H, dk, dv):
    return {"S": 0.3 * rng.standard_normal((B, H, dk, dv)),
            "k_prev": rng.standard_normal((B, H, dk)) / np.sqrt(dk),
            "pos": np.array([[0, 2][: H]] * B, dtype=np.int64)[:, :H] if H <= 2 else np.ones((B, H), np.int64)}


@pytest.mark.parametrize("variant", ONE)
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_g1_torch_forward_is_the_oracle(variant, pairing):
    rng = np.random.default_rng(400 + variant)
    x = inputs(rng, 2, 9, 2, 5, 4, O.is_per_channel(variant))
    carry = carry_for(rng, 2, 2, 5, 4)
    o_n, c_n = O.recurrent(**x, variant=variant, carry=carry, pairing=pairing)
    g = O.recurrent_vjp(**x, variant=variant, do=np.zeros_like(o_n), carry=carry, pairing=pairing)
    assert np.abs(g["o"] - o_n).max() <= 1e-12 * max(1.0, np.abs(o_n).max())
    assert np.abs(g["S"] - c_n["S"]).max() <= 1e-12 * max(1.0, np.abs(c_n["S"]).max())


def _loss(x, variant, do, dS, carry, pairing):
    o, c = O.recurrent(**x, variant=variant, carry=carry, pairing=pairing)
    return (o * do).sum() + (c["S"] * dS).sum()


@pytest.mark.parametrize("variant", ONE)
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_g2_gradients_match_finite_differences(variant, pairing):
    rng = np.random.default_rng(410 + variant)
    B, T, H, dk, dv = 1, 7, 2, 3, 3
    x = inputs(rng, B, T, H, dk, dv, O.is_per_channel(variant))
    carry = carry_for(rng, B, H, dk, dv)
    do = rng.standard_normal((B, T, H, dv))
    dS = rng.standard_normal((B, H, dk, dv))
    g = O.recurrent_vjp(**x, variant=variant, do=do, dS_final=dS, carry=carry, pairing=pairing)
    h = 1e-6
    names = {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "lam": "dlam"}
    for name, gname in names.items():
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (_loss(xp, variant, do, dS, carry, pairing) - _loss(xm, variant, do, dS, carry, pairing)) / (2 * h)
        assert np.abs(fd - g[gname]).max() <= 1e-6 * max(1.0, np.abs(fd).max()), name
    for cname, gname in (("S", "dS_in"), ("k_prev", "dk_prev")):
        fd = np.zeros_like(carry[cname])
        for idx in np.ndindex(carry[cname].shape):
            cp = dict(carry, **{cname: carry[cname].copy()})
            cm = dict(carry, **{cname: carry[cname].copy()})
            cp[cname][idx] += h
            cm[cname][idx] -= h
            fd[idx] = (_loss(x, variant, do, dS, cp, pairing) - _loss(x, variant, do, dS, cm, pairing)) / (2 * h)
        assert np.abs(fd - g[gname]).max() <= 1e-6 * max(1.0, np.abs(fd).max()), cname


def test_g3_clamp_and_missing_pairs_pass_no_gradient():
    rng = np.random.default_rng(420)
    x = inputs(rng, 1, 8, 1, 4, 4, False)
    x["lam"][0, 3, 0] = 1.0          # gamma clamped to eps_gamma
    do = rng.standard_normal((1, 8, 1, 4))
    g = O.recurrent_vjp(**x, variant=O.FALCON_1, do=do)
    assert g["dlam"][0, 3, 0] == 0.0
    assert np.abs(g["dlam"]).sum() > 0
    assert g["dbeta"][0, 0, 0] == 0.0   # fresh sequence: pair 0 does not exist
    assert np.abs(g["dbeta"][0, 1:, 0]).min() > 0
