"""Pins of the backward oracle (oracle/falcon_grad.py).

G1  its torch forward equals the numpy oracle's recurrence (every one-pair
    variant, carries, both pairings), so the function being differentiated
    is the pinned forward
G2  its gradients equal central finite differences of
    L = <o, do> + <S_final, dS_final> for every input, including the carried
    state and key
G3  a clamped decay passes no gradient to lambda, and a step whose pair does
    not exist passes none to beta
G4  the window variants (Falcon-3/3A): G1 and G2 with a carried window ring
    whose slots hold existing and missing pairs (the gradient of every ring
    entry included), and W = 1 gives Falcon-1's / 1A's gradients
G5  closed forms: Falcon-1A without decay and with same-step pairs is causal
    linear attention weighted by eta, o_t = sum_{s<=t} eta_s (q_t . k_s) v_s,
    whose value, query, beta, key, carried-state and decay gradients are
    written out with causal masks; and one Falcon-1 (regression) step, one
    Falcon-2 (per-channel) step and one Falcon-3 (window of two pairs, one of
    them from the carried ring) step from a carried state, every gradient
    derived by hand
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


WIN = [O.FALCON_3, O.FALCON_3A]


def ring_carry(rng, B, H, dk, dv, W, pos):
    """A carry with window ring: pos [H] tokens consumed per head (same for
    every batch row)."""
    c = carry_for(rng, B, H, dk, dv)
    c["pos"] = np.array([pos] * B, dtype=np.int64)
    c["win_x"] = rng.standard_normal((B, H, W - 1, dk)) / np.sqrt(dk)
    c["win_v"] = rng.standard_normal((B, H, W - 1, dv))
    return c


@pytest.mark.parametrize("variant", WIN)
@pytest.mark.parametrize("pairing", ["prefix", "same"])
@pytest.mark.parametrize("W", [2, 4])
def test_g4_window_torch_forward_is_the_oracle(variant, pairing, W):
    rng = np.random.default_rng(430 + variant + 10 * W)
    x = inputs(rng, 2, 9, 3, 5, 4, False)
    carry = ring_carry(rng, 2, 3, 5, 4, W, [0, 2, 7])
    o_n, c_n = O.recurrent(**x, variant=variant, window=W, carry=carry, pairing=pairing)
    g = O.recurrent_vjp(**x, variant=variant, do=np.zeros_like(o_n), carry=carry, pairing=pairing, window=W)
    assert np.abs(g["o"] - o_n).max() <= 1e-12 * max(1.0, np.abs(o_n).max())
    assert np.abs(g["S"] - c_n["S"]).max() <= 1e-12 * max(1.0, np.abs(c_n["S"]).max())


def _loss_w(x, variant, do, dS, carry, pairing, W):
    o, c = O.recurrent(**x, variant=variant, window=W, carry=carry, pairing=pairing)
    return (o * do).sum() + (c["S"] * dS).sum()


@pytest.mark.parametrize("variant", WIN)
@pytest.mark.parametrize("pairing", ["prefix", "same"])
def test_g4_window_gradients_match_finite_differences(variant, pairing):
    rng = np.random.default_rng(440 + variant)
    B, T, H, dk, dv, W = 1, 6, 3, 3, 2, 3
    x = inputs(rng, B, T, H, dk, dv, False)
    carry = ring_carry(rng, B, H, dk, dv, W, [0, 2, 5])
    do = rng.standard_normal((B, T, H, dv))
    dS = rng.standard_normal((B, H, dk, dv))
    g = O.recurrent_vjp(**x, variant=variant, do=do, dS_final=dS, carry=carry, pairing=pairing, window=W)
    h = 1e-6
    L = lambda xx, cc: _loss_w(xx, variant, do, dS, cc, pairing, W)
    for name, gname in {"q": "dq", "k": "dk", "v": "dv", "beta": "dbeta", "lam": "dlam"}.items():
        fd = np.zeros_like(x[name])
        for idx in np.ndindex(x[name].shape):
            xp = {kk: vv.copy() for kk, vv in x.items()}
            xm = {kk: vv.copy() for kk, vv in x.items()}
            xp[name][idx] += h
            xm[name][idx] -= h
            fd[idx] = (L(xp, carry) - L(xm, carry)) / (2 * h)
        assert np.abs(fd - g[gname]).max() <= 1e-6 * max(1.0, np.abs(fd).max()), name
    for cname, gname in (("S", "dS_in"), ("k_prev", "dk_prev"), ("win_x", "dwin_x"), ("win_v", "dwin_v")):
        fd = np.zeros_like(carry[cname])
        for idx in np.ndindex(carry[cname].shape):
            cp = dict(carry, **{cname: carry[cname].copy()})
            cm = dict(carry, **{cname: carry[cname].copy()})
            cp[cname][idx] += h
            cm[cname][idx] -= h
            fd[idx] = (L(x, cp) - L(x, cm)) / (2 * h)
        assert np.abs(fd - g[gname]).max() <= 1e-6 * max(1.0, np.abs(fd).max()), cname
    # ring slots of pairs that do not exist (global index below the first pair) get nothing
    first = 1 if pairing == "prefix" else 0
    for hh, p0 in enumerate([0, 2, 5]):
        for p in range(p0 - (W - 1), p0):
            if p < first:
                s = p % (W - 1)
                assert not g["dwin_x"][0, hh, s].any() and not g["dwin_v"][0, hh, s].any()


@pytest.mark.parametrize("pair", [(O.FALCON_3, O.FALCON_1), (O.FALCON_3A, O.FALCON_1A)])
def test_g4_window_one_is_the_one_pair_gradient(pair):
    rng = np.random.default_rng(450 + pair[0])
    x = inputs(rng, 1, 8, 2, 4, 3, False)
    carry = carry_for(rng, 1, 2, 4, 3)
    do = rng.standard_normal((1, 8, 2, 3))
    g3 = O.recurrent_vjp(**x, variant=pair[0], do=do, carry=carry, window=1)
    g1 = O.recurrent_vjp(**x, variant=pair[1], do=do, carry=carry)
    for n in ("dq", "dk", "dv", "dbeta", "dlam", "dS_in", "dk_prev"):
        assert np.abs(g3[n] - g1[n]).max() <= 1e-13 * max(1.0, np.abs(g1[n]).max()), n


def test_g5_linear_attention_closed_forms():
    """lambda = 0 gives gamma = 1 (no decay), and Falcon-1A's additive write
    with same-step pairs accumulates S_t = sum_{s<=t} eta_s k_s v_s^T, so
    o_t = S_t^T q_t = sum_{s<=t} eta_s (q_t . k_s) v_s with eta_s =
    beta_s / (eps + |k_s|^2) [FW Falcon 家族; JC Falcon家族六个变体各管一段].
    For L = <o, dO>, with A_ts = (q_t . k_s) for s <= t (else 0):
      dv_s = eta_s sum_t A_ts do_t,          dq_t = sum_{s<=t} eta_s (do_t . v_s) k_s,
      dbeta_s = sum_t A_ts (v_s . do_t) / (eps + |k_s|^2)."""
    rng = np.random.default_rng(71)
    B, T, H, d = 1, 12, 2, 5
    x = inputs(rng, B, T, H, d, d, False)
    x["lam"] = np.zeros((B, T, H))
    do = rng.standard_normal((B, T, H, d))
    eps = 1e-6
    g = O.recurrent_vjp(x["q"], x["k"], x["v"], x["beta"], x["lam"], O.FALCON_1A, do, None, eps, 1e-3,
                        pairing="same")
    for h in range(H):
        q, k, v, dO = (a[0, :, h] for a in (x["q"], x["k"], x["v"], do))
        den = eps + (k * k).sum(-1)
        eta = x["beta"][0, :, h] / den
        A = np.tril(q @ k.T)                       # A[t, s] = q_t . k_s, s <= t
        dv = eta[:, None] * (A.T @ dO)
        dq = np.tril(dO @ v.T) @ (eta[:, None] * k)
        dbeta = (A * (dO @ v.T)).sum(0) / den
        assert np.allclose(g["dv"][0, :, h], dv, rtol=1e-10, atol=1e-12)
        assert np.allclose(g["dq"][0, :, h], dq, rtol=1e-10, atol=1e-12)
        assert np.allclose(g["dbeta"][0, :, h], dbeta, rtol=1e-10, atol=1e-12)


def test_g5_linear_attention_closed_forms_keys_state_decay():
    """The same case with a carried state S_in (o_t gains S_in^T q_t) and an
    end-state cotangent dS_final (S_T = S_in + sum_s eta_s k_s v_s^T): the key
    gradient, with the eta term,
      dk_s = eta_s (sum_t (v_s . do_t) q_t + dS_final v_s)
             - 2 beta_s k_s / (eps + |k_s|^2)^2 (sum_t A_ts (v_s . do_t) + k_s^T dS_final v_s),
    the carried state's gradient is dS_in = sum_t q_t do_t^T + dS_final, and
    the decay gradient at gamma = 1 (inside the clamp) is dlambda_t = -dgamma_t,
      dgamma_t = <sum_{u>=t} q_u do_u^T + dS_final, S_{t-1}>,
      S_{t-1} = S_in + sum_{s<t} eta_s k_s v_s^T."""
    rng = np.random.default_rng(72)
    B, T, H, d = 1, 10, 1, 4
    x = inputs(rng, B, T, H, d, d, False)
    x["lam"] = np.zeros((B, T, H))
    do = rng.standard_normal((B, T, H, d))
    dSf = rng.standard_normal((B, H, d, d))
    S_in = 0.5 * rng.standard_normal((B, H, d, d))
    eps = 1e-6
    g = O.recurrent_vjp(x["q"], x["k"], x["v"], x["beta"], x["lam"], O.FALCON_1A, do, dSf, eps, 1e-3,
                        carry={"S": S_in}, pairing="same")
    q, k, v, dO = (a[0, :, 0] for a in (x["q"], x["k"], x["v"], do))
    beta = x["beta"][0, :, 0]
    den = eps + (k * k).sum(-1)
    eta = beta / den
    A = np.tril(q @ k.T)
    VD = dO @ v.T                                   # VD[t, s] = do_t . v_s
    Sv = v @ dSf[0, 0].T                             # Sv[s] = dS_final v_s
    kSv = (k * Sv).sum(-1)                           # k_s^T dS_final v_s
    dk = (eta[:, None] * (np.tril(VD).T @ q + Sv)
          - (2 * beta / den ** 2)[:, None] * k * ((A * VD).sum(0) + kSv)[:, None])
    assert np.allclose(g["dk"][0, :, 0], dk, rtol=1e-9, atol=1e-11)
    assert np.allclose(g["dS_in"][0, 0], q.T @ dO + dSf[0, 0], rtol=1e-10, atol=1e-12)
    dgam = np.zeros(T)
    for t in range(T):
        S_prev = S_in[0, 0] + sum(eta[s] * np.outer(k[s], v[s]) for s in range(t))
        dS_t = q[t:].T @ dO[t:] + dSf[0, 0]
        dgam[t] = (dS_t * S_prev).sum()
    assert np.allclose(g["dlam"][0, :, 0], -dgam, rtol=1e-9, atol=1e-11)


def test_g5_one_regression_step_closed_forms():
    """One Falcon-1 step from a carried state, same-step pair x = k_0 [FW
    Falcon 家族; JC Falcon家族六个变体各管一段]: with gamma the clamped decay,
    eta = beta / (eps + |x|^2), r = v - gamma S0^T x,
      S1 = gamma S0 + eta x r^T = gamma (I - eta x x^T) S0 + eta x v^T,  o = S1^T q,
    and G = dS1 = q do^T + dS_final, the gradients written out by hand:
      dq = S1 do,  dv = eta G^T x,  dS0 = gamma (I - eta x x^T) G,
      dgamma = <G, (I - eta x x^T) S0>  (dlambda = -dgamma inside the clamp),
      dbeta = x^T G r / (eps + |x|^2),
      dk = eta G v - eta gamma (G S0^T x + S0 G^T x) - 2 beta x (x^T G r) / (eps + |x|^2)^2."""
    rng = np.random.default_rng(73)
    d = 5
    x = inputs(rng, 1, 1, 1, d, d, False)
    do = rng.standard_normal((1, 1, 1, d))
    dSf = rng.standard_normal((1, 1, d, d))
    S0 = 0.5 * rng.standard_normal((1, 1, d, d))
    eps, eps_g = 1e-6, 1e-3
    g = O.recurrent_vjp(x["q"], x["k"], x["v"], x["beta"], x["lam"], O.FALCON_1, do, dSf, eps, eps_g,
                        carry={"S": S0}, pairing="same")
    q, k, v, dO = (a[0, 0, 0] for a in (x["q"], x["k"], x["v"], do))
    beta, lam, S, Gf = x["beta"][0, 0, 0], x["lam"][0, 0, 0], S0[0, 0], dSf[0, 0]
    gamma = min(max(1.0 - lam, eps_g), 1.0)
    assert eps_g < 1.0 - lam < 1.0   # inside the clamp: the gradient passes
    den = eps + k @ k
    eta = beta / den
    r = v - gamma * (S.T @ k)
    P = np.eye(d) - eta * np.outer(k, k)
    S1 = gamma * S + eta * np.outer(k, r)
    G = np.outer(q, dO) + Gf
    want = {
        "dq": S1 @ dO,
        "dv": eta * (G.T @ k),
        "dS_in": gamma * (P @ G),
        "dlam": -np.sum(G * (P @ S)),
        "dbeta": (k @ G @ r) / den,
        "dk": eta * (G @ v) - eta * gamma * (G @ S.T @ k + S @ G.T @ k) - 2 * beta * k * (k @ G @ r) / den ** 2,
    }
    got = {"dq": g["dq"][0, 0, 0], "dv": g["dv"][0, 0, 0], "dS_in": g["dS_in"][0, 0], "dlam": g["dlam"][0, 0, 0],
           "dbeta": g["dbeta"][0, 0, 0], "dk": g["dk"][0, 0, 0]}
    for n, w_ in want.items():
        assert np.allclose(got[n], w_, rtol=1e-10, atol=1e-12), n


def test_g5_one_per_channel_step_closed_forms():
    """One Falcon-2 step (per-channel step size, eta_j = beta_j / (eps + |x|^2)
    for value channel j) from a carried state, same-step pair x = k_0:
      S1 = gamma S0 + x (eta (.) (v - gamma S0^T x))^T = gamma (S0 - x x^T S0 D) + x v^T D,
    D = diag(eta), G = q do^T + dS_final, r = v - gamma S0^T x:
      dq = S1 do,  dv = D G^T x,  dS0 = gamma (G - x x^T G D),
      dgamma = <G, S0 - x x^T S0 D>,  d eta_j = (G^T x)_j r_j,  dbeta_j = d eta_j / (eps + |x|^2),
      dk = G D v - gamma (G D S0^T x + S0 D G^T x) - 2 x (sum_j d eta_j beta_j) / (eps + |x|^2)^2."""
    rng = np.random.default_rng(74)
    d = 5
    x = inputs(rng, 1, 1, 1, d, d, True)
    do = rng.standard_normal((1, 1, 1, d))
    dSf = rng.standard_normal((1, 1, d, d))
    S0 = 0.5 * rng.standard_normal((1, 1, d, d))
    eps, eps_g = 1e-6, 1e-3
    g = O.recurrent_vjp(x["q"], x["k"], x["v"], x["beta"], x["lam"], O.FALCON_2, do, dSf, eps, eps_g,
                        carry={"S": S0}, pairing="same")
    q, k, v, dO = (a[0, 0, 0] for a in (x["q"], x["k"], x["v"], do))
    beta, lam, S, Gf = x["beta"][0, 0, 0], x["lam"][0, 0, 0], S0[0, 0], dSf[0, 0]
    gamma = min(max(1.0 - lam, eps_g), 1.0)
    assert eps_g < 1.0 - lam < 1.0
    den = eps + k @ k
    eta = beta / den
    D = np.diag(eta)
    r = v - gamma * (S.T @ k)
    S1 = gamma * S + np.outer(k, eta * r)
    G = np.outer(q, dO) + Gf
    deta = (G.T @ k) * r
    xx = np.outer(k, k)
    want = {
        "dq": S1 @ dO,
        "dv": D @ G.T @ k,
        "dS_in": gamma * (G - xx @ G @ D),
        "dlam": -np.sum(G * (S - xx @ S @ D)),
        "dbeta": deta / den,
        "dk": G @ D @ v - gamma * (G @ D @ S.T @ k + S @ D @ G.T @ k) - 2 * k * (deta @ beta) / den ** 2,
    }
    got = {"dq": g["dq"][0, 0, 0], "dv": g["dv"][0, 0, 0], "dS_in": g["dS_in"][0, 0], "dlam": g["dlam"][0, 0, 0],
           "dbeta": g["dbeta"][0, 0, 0], "dk": g["dk"][0, 0, 0]}
    for n, w_ in want.items():
        assert np.allclose(got[n], w_, rtol=1e-10, atol=1e-12), n


@pytest.mark.parametrize("variant", [O.FALCON_3, O.FALCON_3A])
def test_g5_one_window_step_closed_forms(variant):
    """One Falcon-3 step with W = 2 and same-step pairs [FW Falcon 家族; JC
    Falcon家族六个变体各管一段]: the window holds the carried ring pair a
    (x_a, v_a) and the step's own pair b (k_0, v_0), both existing (pos = 3),
    n = 2, e = (|x_a|^2 + |x_b|^2) / 2, eta = beta / (eps + e), c = eta / n,
    r_i = v_i - gamma S0^T x_i, and
      S1 = gamma S0 + c sum_i x_i r_i^T = gamma (I - c X) S0 + c sum_i x_i v_i^T,  X = sum_i x_i x_i^T.
    With G = q do^T + dS_final and dc = sum_i x_i^T G r_i:
      dq = S1 do,  dv_i = c G^T x_i,  dS0 = gamma (I - c X) G,
      dgamma = <G, (I - c X) S0>,  dbeta = dc / (n (eps + e)),
      dx_i = c (G r_i - gamma S0 G^T x_i) - (dc / n) eta / (eps + e) (2 x_i / n),
    dk_0 = dx_b and the ring entry's gradients dx_a, dv_a.  Falcon-3A writes
    additively: r_i = v_i, so the gamma S0^T x_i terms drop (dS0 = gamma G,
    dgamma = <G, S0>, dx_i = c G v_i + the e term)."""
    rng = np.random.default_rng(75)
    d, W = 4, 2
    x = inputs(rng, 1, 1, 1, d, d, False)
    do = rng.standard_normal((1, 1, 1, d))
    dSf = rng.standard_normal((1, 1, d, d))
    S0 = 0.5 * rng.standard_normal((1, 1, d, d))
    xa = rng.standard_normal((1, 1, W - 1, d)) / np.sqrt(d)
    va = rng.standard_normal((1, 1, W - 1, d))
    eps, eps_g = 1e-6, 1e-3
    carry = {"S": S0, "pos": np.array([[3]], dtype=np.int64), "win_x": xa, "win_v": va}
    g = O.recurrent_vjp(x["q"], x["k"], x["v"], x["beta"], x["lam"], variant, do, dSf, eps, eps_g,
                        carry=carry, pairing="same", window=W)
    add = variant == O.FALCON_3A
    q, kb, vb, dO = (a[0, 0, 0] for a in (x["q"], x["k"], x["v"], do))
    beta, lam, S, Gf = x["beta"][0, 0, 0], x["lam"][0, 0, 0], S0[0, 0], dSf[0, 0]
    pa, qa = xa[0, 0, 0], va[0, 0, 0]
    gamma = min(max(1.0 - lam, eps_g), 1.0)
    assert eps_g < 1.0 - lam < 1.0
    n = 2.0
    e = (pa @ pa + kb @ kb) / n
    eta = beta / (eps + e)
    c = eta / n
    X = np.zeros((d, d)) if add else np.outer(pa, pa) + np.outer(kb, kb)  # the residual's S0 term
    I = np.eye(d)
    sg = 0.0 if add else gamma
    ra, rb = qa - sg * (S.T @ pa), vb - sg * (S.T @ kb)
    S1 = gamma * (I - c * X) @ S + c * (np.outer(pa, qa) + np.outer(kb, vb))
    G = np.outer(q, dO) + Gf
    dc = pa @ G @ ra + kb @ G @ rb
    de = -(dc / n) * eta / (eps + e)
    dx = lambda xi, ri: c * (G @ ri - sg * S @ G.T @ xi) + de * 2 * xi / n
    want = {
        "dq": S1 @ dO,
        "dv": c * (G.T @ kb),
        "dS_in": gamma * (I - c * X) @ G,
        "dlam": -np.sum(G * ((I - c * X) @ S)),
        "dbeta": dc / (n * (eps + e)),
        "dk": dx(kb, rb),
        "dwin_x": dx(pa, ra),
        "dwin_v": c * (G.T @ pa),
    }
    got = {"dq": g["dq"][0, 0, 0], "dv": g["dv"][0, 0, 0], "dS_in": g["dS_in"][0, 0], "dlam": g["dlam"][0, 0, 0],
           "dbeta": g["dbeta"][0, 0, 0], "dk": g["dk"][0, 0, 0], "dwin_x": g["dwin_x"][0, 0, 0],
           "dwin_v": g["dwin_v"][0, 0, 0]}
    for nme, w_ in want.items():
        assert np.allclose(got[nme], w_, rtol=1e-10, atol=1e-12), nme
