"""Pins of the CPU oracle against what the Falcon pages and the mathematics fix.

None of these re-types the oracle's own formula: each checks it against an
independent fact (a hand-derived example, a closed form, an invariant that
follows from the update, another algebraic form of the same method, or a
special case that reduces to a textbook rule).

P1  three-form equivalence (recurrent = masked-parallel = chunked)
    [Falcon 家族重新对齐 fast-weight 记忆, 三种等价形式]
P2  Falcon-1A without decay is causal denominator-free linear attention with
    prefix-shifted keys [same page, 三种等价形式]
P3  NLMS step: exact residual identity and per-step loss decrease
    [给记忆装一个“及时纠错”的开关, 把记忆更新变成一次梯度下降]
P4  Falcon-3 window averaging: W = 1 is Falcon-1, identical pairs give the
    Falcon-1 update for any W, the step operator is bounded by beta
    [same page, Falcon家族六个变体各管一段 and 写在后面]
P5  positive-decay clamp keeps every log-decay finite [same page, 正衰减钳制]
P6  closed forms: hand-derived scalar sequences, exact orthonormal retrieval
P7  variant reductions: Falcon-2 with equal channels is Falcon-1 (and 2A is 1A)
P8  same-step pairing (the ablation of the prefix alignment): the three forms
    agree; it equals the prefix alignment fed the next key; with unit step it
    is the classical delta rule, which reads back the value just written
    [Falcon 家族重新对齐 fast-weight 记忆, 本质; 给记忆装一个“及时纠错”的开关,
    一个被忽略的时间差]
"""

import json
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden", "scalar_nlms.json")


def rand_inputs(rng, B, T, H, dk, dv, per_channel=False, gamma_mu=3.0, gamma_sd=1.0):
    q = rng.standard_normal((B, T, H, dk))
    q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, H, dv))
    bshape = (B, T, H, dv) if per_channel else (B, T, H)
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(bshape)))
    gamma = 1.0 / (1.0 + np.exp(-(gamma_mu + gamma_sd * rng.standard_normal((B, T, H)))))
    return dict(q=q, k=k, v=v, beta=beta, lam=1.0 - gamma)


def rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


ALL = [O.FALCON_1, O.FALCON_1A, O.FALCON_2, O.FALCON_2A, O.FALCON_3, O.FALCON_3A]


# ---------------------------------------------------------------- P1
@pytest.mark.parametrize("variant", ALL)
@pytest.mark.parametrize("chunk", [1, 4, 16, 61])
def test_p1_three_forms_agree(variant, chunk):
    rng = np.random.default_rng(100 + variant)
    W = 3 if O.is_windowed(variant) else 1
    x = rand_inputs(rng, 2, 61, 2, 8, 6, O.is_per_channel(variant))  # T=61: ragged
    o_r, c_r = O.recurrent(**x, variant=variant, window=W)
    o_m, S_m = O.masked_parallel(**x, variant=variant, window=W)
    o_c, c_c = O.chunked(**x, variant=variant, window=W, chunk=chunk)
    assert rel(o_m, o_r) <= 1e-10
    assert rel(S_m, c_r["S"]) <= 1e-10
    assert rel(o_c, o_r) <= 1e-10
    assert rel(c_c["S"], c_r["S"]) <= 1e-10


def test_p1_tiny_reference_case():
    """The 1x64x1, d=16, chunk=16 fp32 case: all three forms, sub-second."""
    from workloads import TINY_F1, make_inputs
    x = {k: v.double().numpy() for k, v in make_inputs(TINY_F1).items()}
    o_r, c_r = O.recurrent(**x, variant=O.FALCON_1)
    o_m, S_m = O.masked_parallel(**x, variant=O.FALCON_1)
    o_c, c_c = O.chunked(**x, variant=O.FALCON_1, chunk=16)
    assert rel(o_m, o_r) <= 1e-10 and rel(o_c, o_r) <= 1e-10
    assert rel(S_m, c_r["S"]) <= 1e-10 and rel(c_c["S"], c_r["S"]) <= 1e-10


@pytest.mark.parametrize("variant", ALL)
def test_p1_chunked_with_carry(variant):
    """The chunked form from a carried state equals the recurrence."""
    rng = np.random.default_rng(7 + variant)
    W = 4 if O.is_windowed(variant) else 1
    x = rand_inputs(rng, 2, 23, 2, 6, 5, O.is_per_channel(variant))
    carry = {
        "S": rng.standard_normal((2, 2, 6, 5)) * 0.4,
        "k_prev": rng.standard_normal((2, 2, 6)) * 0.5,
        "pos": np.array([[2, 9], [0, 1]]),
    }
    if W > 1:
        carry["win_x"] = rng.standard_normal((2, 2, W - 1, 6)) * 0.5
        carry["win_v"] = rng.standard_normal((2, 2, W - 1, 5))
    o_r, c_r = O.recurrent(**x, variant=variant, window=W, carry=carry)
    o_c, c_c = O.chunked(**x, variant=variant, window=W, chunk=8, carry=carry)
    assert rel(o_c, o_r) <= 1e-10
    for key in c_r:
        assert np.abs(c_c[key] - c_r[key]).max() <= 1e-10 * max(1.0, np.abs(c_r[key]).max())


@pytest.mark.parametrize("variant", ALL)
def test_carry_round_trip(variant):
    """Splitting a sequence and carrying the state gives the same result."""
    rng = np.random.default_rng(11 + variant)
    W = 3 if O.is_windowed(variant) else 1
    x = rand_inputs(rng, 1, 30, 2, 5, 4, O.is_per_channel(variant))
    o_full, c_full = O.recurrent(**x, variant=variant, window=W)
    a = {k: v[:, :13] for k, v in x.items()}
    b = {k: v[:, 13:] for k, v in x.items()}
    o_a, c_a = O.recurrent(**a, variant=variant, window=W)
    o_b, c_b = O.recurrent(**b, variant=variant, window=W, carry=c_a)
    assert np.abs(np.concatenate([o_a, o_b], 1) - o_full).max() <= 1e-12
    for key in c_full:
        assert np.abs(c_b[key] - c_full[key]).max() <= 1e-12


# ---------------------------------------------------------------- P2
def test_p2_falcon1a_no_decay_is_linear_attention():
    rng = np.random.default_rng(2)
    B, T, H, dk, dv = 1, 40, 2, 7, 5
    x = rand_inputs(rng, B, T, H, dk, dv)
    x["lam"] = np.zeros((B, T, H))
    eps = 1e-6
    # beta_s := eps + ||x_s||^2 makes eta_s = 1: plain linear attention.
    xs = np.zeros((B, T, H, dk))
    xs[:, 1:] = x["k"][:, :-1]
    x["beta"] = eps + (xs ** 2).sum(-1)
    o, _ = O.recurrent(**x, variant=O.FALCON_1A, eps=eps)
    brute = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            for t in range(T):
                for s in range(1, t + 1):   # pair s = (k_{s-1}, v_s); s = 0 has no key
                    brute[b, t, h] += (x["q"][b, t, h] @ x["k"][b, s - 1, h]) * x["v"][b, s, h]
    assert np.abs(o - brute).max() <= 1e-12


def test_p2_falcon1a_general_eta_is_masked_linear_attention():
    """With any beta: (Q X^T (.) M_eta) V where M_ts = eta_s [1 <= s <= t]."""
    rng = np.random.default_rng(3)
    B, T, H, dk, dv = 1, 33, 1, 6, 4
    x = rand_inputs(rng, B, T, H, dk, dv)
    x["lam"] = np.zeros((B, T, H))
    o, _ = O.recurrent(**x, variant=O.FALCON_1A)
    q, k, v, beta = x["q"][0, :, 0], x["k"][0, :, 0], x["v"][0, :, 0], x["beta"][0, :, 0]
    Xs = np.vstack([np.zeros((1, dk)), k[:-1]])
    eta = beta / (1e-6 + (Xs ** 2).sum(-1))
    eta[0] = 0.0
    M = np.tril(np.ones((T, T))) * eta[None, :]
    assert np.abs(o[0, :, 0] - ((q @ Xs.T) * M) @ v).max() <= 1e-12


# ---------------------------------------------------------------- P3
@pytest.mark.parametrize("variant", [O.FALCON_1, O.FALCON_2])
def test_p3_nlms_residual_identity_and_decrease(variant):
    rng = np.random.default_rng(5)
    B, T, H, dk, dv = 2, 25, 2, 6, 5
    per_ch = O.is_per_channel(variant)
    x = rand_inputs(rng, B, T, H, dk, dv, per_ch)
    x["k"] = x["k"] * rng.uniform(0.3, 3.0, size=(B, T, H, 1))  # energies != 1
    o, _, tr = O.recurrent(**x, variant=variant, return_trace=True)
    for t in range(1, T):
        xt = x["k"][:, t - 1]                       # [B, H, dk]
        vt = x["v"][:, t]
        S = tr["S"][t]
        r = tr["r"][t]                               # v_t - Z_t^T x_t
        after = vt - np.einsum("bhk,bhkv->bhv", xt, S)
        n2 = (xt ** 2).sum(-1)
        bt = x["beta"][:, t]
        if per_ch:
            eta = bt / (1e-6 + n2[..., None])
            factor = 1.0 - eta * n2[..., None]
        else:
            eta = bt / (1e-6 + n2)
            factor = (1.0 - eta * n2)[..., None]
        assert np.abs(after - factor * r).max() <= 1e-12
        # 0 < eta ||x||^2 < beta < 1: strict decrease of every residual entry
        assert np.all(np.abs(after) <= np.abs(r) + 1e-15)
        assert np.all((after ** 2).sum(-1) < (r ** 2).sum(-1))


def test_p3_exact_fit_with_unit_beta():
    rng = np.random.default_rng(6)
    x = rand_inputs(rng, 1, 12, 1, 4, 3)
    x["beta"] = np.ones_like(x["beta"])
    eps = 1e-9
    _, _, tr = O.recurrent(**x, variant=O.FALCON_1, eps=eps, return_trace=True)
    for t in range(1, 12):
        xt = x["k"][0, t - 1, 0]
        pred = xt @ tr["S"][t][0, 0]
        assert np.abs(pred - x["v"][0, t, 0]).max() <= 1e-7


def test_p3_window_loss_decreases():
    """Falcon-3: the window-averaged squared loss drops at every step."""
    rng = np.random.default_rng(8)
    W = 4
    x = rand_inputs(rng, 1, 30, 1, 5, 3)
    x["k"] = x["k"] * rng.uniform(0.5, 2.0, size=(1, 30, 1, 1))
    _, _, tr = O.recurrent(**x, variant=O.FALCON_3, window=W, return_trace=True)
    X, V, valid, _ = O.build_pairs(x["k"], x["v"], W)
    for t in range(1, 30):
        idx = [i for i in range(t, t + W) if valid[0, 0, i]]
        def loss(S):
            return sum(((V[0, 0, i] - X[0, 0, i] @ S) ** 2).sum() for i in idx) / (2 * len(idx))
        assert loss(tr["S"][t][0, 0]) < loss(tr["Z"][t][0, 0])


# ---------------------------------------------------------------- P4
def test_p4_window_one_is_falcon1():
    rng = np.random.default_rng(9)
    x = rand_inputs(rng, 2, 27, 2, 6, 4)
    o1, c1 = O.recurrent(**x, variant=O.FALCON_1)
    o3, c3 = O.recurrent(**x, variant=O.FALCON_3, window=1)
    assert np.abs(o1 - o3).max() == 0.0 and np.abs(c1["S"] - c3["S"]).max() == 0.0
    o1a, _ = O.recurrent(**x, variant=O.FALCON_1A)
    o3a, _ = O.recurrent(**x, variant=O.FALCON_3A, window=1)
    assert np.abs(o1a - o3a).max() == 0.0


@pytest.mark.parametrize("W", [2, 4, 8])
@pytest.mark.parametrize("pair", [(O.FALCON_3, O.FALCON_1), (O.FALCON_3A, O.FALCON_1A)])
def test_p4_identical_pairs_give_falcon1_update(W, pair):
    """Averaging (not summing): W copies of one pair move the state exactly
    as one copy does, for every window size; for the regression window
    (Falcon-3 against Falcon-1) and the additive one (Falcon-3A against
    Falcon-1A)."""
    windowed, single = pair
    rng = np.random.default_rng(10)
    B, T, H, dk, dv = 1, 20, 1, 6, 4
    x = rand_inputs(rng, B, T, H, dk, dv)
    x["k"][:] = x["k"][:, :1]
    x["v"][:] = x["v"][:, :1]
    o1, c1 = O.recurrent(**x, variant=single)
    o3, c3 = O.recurrent(**x, variant=windowed, window=W)
    assert rel(o3, o1) <= 1e-12 and rel(c3["S"], c1["S"]) <= 1e-12


@pytest.mark.parametrize("W", [2, 3, 8])
def test_p4_falcon3a_is_window_masked_linear_attention(W):
    """Falcon-3A, written out by brute force from the additive window write
    [给记忆装一个“及时纠错”的开关, Falcon家族六个变体各管一段]: with the decay
    products D(t, s) = prod_{s < u <= t} gamma_u, every step s writes
    (eta_s / n_s) x_j v_j^T for each existing pair j of its window, so
    o_t = sum_{s <= t} D(t, s) (eta_s / n_s) sum_{j in W(s)} (q_t . x_j) v_j,
    eta_s = beta_s / (eps + mean_{j in W(s)} |x_j|^2).  Keys of varied
    energy, so the window-average energy is not a constant."""
    rng = np.random.default_rng(40 + W)
    B, T, H, dk, dv = 1, 29, 2, 5, 3
    x = rand_inputs(rng, B, T, H, dk, dv)
    x["k"] = x["k"] * rng.uniform(0.3, 2.5, size=(B, T, H, 1))
    eps, eg = 1e-6, 1e-3
    o, c = O.recurrent(**x, variant=O.FALCON_3A, window=W, eps=eps, eps_gamma=eg)
    gam = np.clip(1.0 - x["lam"], eg, 1.0)
    brute = np.zeros((B, T, H, dv))
    Sb = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            keys = {j: x["k"][b, j - 1, h] for j in range(1, T)}  # pair j = (k_{j-1}, v_j), j >= 1
            for t in range(T):
                for s in range(t + 1):
                    win = [j for j in range(s - W + 1, s + 1) if j >= 1]
                    if not win:
                        continue
                    e = np.mean([keys[j] @ keys[j] for j in win])
                    coef = x["beta"][b, s, h] / (eps + e) / len(win)
                    D = np.prod(gam[b, s + 1:t + 1, h])
                    for j in win:
                        brute[b, t, h] += D * coef * (x["q"][b, t, h] @ keys[j]) * x["v"][b, j, h]
                        if t == T - 1:
                            Sb[b, h] += D * coef * np.outer(keys[j], x["v"][b, j, h])
    assert np.abs(o - brute).max() <= 1e-12 * max(1.0, np.abs(brute).max())
    assert np.abs(c["S"] - Sb).max() <= 1e-12 * max(1.0, np.abs(Sb).max())


def test_p4_planted_sum_instead_of_average_is_caught(monkeypatch):
    """Plant the 'sum over the window' mistake in the oracle: the identical-
    pairs pin must fail, its update growing with W."""
    import oracle.falcon as F
    real = F.step_coefficients

    def summed(beta_t, x_win, valid_win, eps, per_channel):
        n = np.maximum(valid_win.sum(-1), 1)
        c = real(beta_t, x_win, valid_win, eps, per_channel)
        return c * (n[..., None, None] if per_channel else n[..., None])

    rng = np.random.default_rng(10)
    x = rand_inputs(rng, 1, 20, 1, 6, 4)
    x["k"][:] = x["k"][:, :1]
    x["v"][:] = x["v"][:, :1]
    o1, _ = F.recurrent(**x, variant=O.FALCON_1)
    monkeypatch.setattr(F, "step_coefficients", summed)
    o3, _ = F.recurrent(**x, variant=O.FALCON_3A, window=8)
    o1a, _ = F.recurrent(**x, variant=O.FALCON_1A)
    assert rel(o3, o1a) > 0.5


@pytest.mark.parametrize("W", [2, 5, 8])
def test_p4_step_operator_bounded_by_beta(W):
    """||(eta_t/n_t) sum_j x_j x_j^T||_2 <= beta_t for every window size."""
    rng = np.random.default_rng(12)
    x = rand_inputs(rng, 1, 40, 1, 6, 3)
    x["k"] = x["k"] * rng.uniform(0.2, 4.0, size=(1, 40, 1, 1))
    X, V, valid, _ = O.build_pairs(x["k"], x["v"], W)
    for t in range(40):
        xw = X[0, 0, t:t + W]
        mw = valid[0, 0, t:t + W].astype(float)
        c = O.step_coefficients(x["beta"][0, t, 0], xw, mw, 1e-6, False)
        op = (xw * c[:, None]).T @ xw
        assert np.linalg.norm(op, 2) <= x["beta"][0, t, 0] + 1e-12


# ---------------------------------------------------------------- P5
def test_p5_clamp_keeps_log_decay_finite():
    rng = np.random.default_rng(13)
    B, T, H = 1, 300, 2
    x = rand_inputs(rng, B, T, H, 8, 8, gamma_mu=4.0, gamma_sd=0.5)
    forced = rng.random((B, T, H)) < 0.05
    x["lam"] = np.where(forced, 1.0, x["lam"])
    eg = 1e-3
    g = O.decay_factor(x["lam"], eg)
    assert np.all(np.log(g) >= np.log(eg)) and np.all(np.isfinite(np.log(g)))
    o, c, tr = O.recurrent(**x, variant=O.FALCON_1, eps_gamma=eg, return_trace=True)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(c["S"]))
    # right after a clamped position the shrunk state is eps_gamma * S_{t-1}
    for t in range(1, T):
        for h in range(H):
            if forced[0, t, h]:
                assert np.allclose(tr["Z"][t][0, h], eg * tr["S"][t - 1][0, h], rtol=0, atol=1e-15)
    o_m, _ = O.masked_parallel(**{k: v[:, :120] for k, v in x.items()}, variant=O.FALCON_1,
                               eps_gamma=eg)
    assert np.all(np.isfinite(o_m))
    o_c, _ = O.chunked(**x, variant=O.FALCON_1, chunk=64, eps_gamma=eg)
    assert rel(o_c, o) <= 1e-10


# ---------------------------------------------------------------- P6
def _gold_inputs():
    g = json.load(open(GOLD))
    i = g["inputs"]
    sh = lambda a: np.array(a, dtype=np.float64).reshape(1, -1, 1, 1)
    x = dict(q=sh(i["q"]), k=sh(i["k"]), v=sh(i["v"]), beta=sh(i["beta"])[..., 0],
             lam=sh(i["lam"])[..., 0])
    return g, x, i["eps"], i["eps_gamma"]


@pytest.mark.parametrize("key,variant,W", [("falcon1", O.FALCON_1, 1),
                                           ("falcon1a", O.FALCON_1A, 1),
                                           ("falcon3_w2", O.FALCON_3, 2)])
def test_p6_hand_derived_scalar_sequences(key, variant, W):
    g, x, eps, eg = _gold_inputs()
    exp = g["expected"][key]
    for form in ("recurrent", "chunked", "masked"):
        if form == "recurrent":
            o, c = O.recurrent(**x, variant=variant, window=W, eps=eps, eps_gamma=eg)
            S = c["S"]
        elif form == "chunked":
            o, c = O.chunked(**x, variant=variant, window=W, chunk=2, eps=eps, eps_gamma=eg)
            S = c["S"]
        else:
            o, S = O.masked_parallel(**x, variant=variant, window=W, eps=eps, eps_gamma=eg)
        assert np.allclose(o.reshape(-1), exp["o"], rtol=0, atol=1e-15), form
        assert abs(S.reshape(-1)[0] - exp["S_final"]) <= 1e-15, form
    o, c = O.recurrent(**x, variant=variant, window=W, eps=eps, eps_gamma=eg)
    if "k_prev" in exp:
        assert c["k_prev"].reshape(-1)[0] == exp["k_prev"] and int(c["pos"].reshape(-1)[0]) == exp["pos"]
    if "win_x" in exp:
        assert c["win_x"].reshape(-1).tolist() == exp["win_x"]
        assert c["win_v"].reshape(-1).tolist() == exp["win_v"]


def test_p6_orthonormal_keys_exact_retrieval():
    """Classical delta rule: with gamma = 1, beta = 1, eps -> 0 and orthonormal
    keys, the state stores every pair exactly (S^T x_j = v_j)."""
    rng = np.random.default_rng(14)
    dk, dv = 8, 5
    Qm, _ = np.linalg.qr(rng.standard_normal((dk, dk)))
    keys = Qm.T                                   # rows orthonormal
    T = dk + 1
    k = np.zeros((1, T, 1, dk))
    k[0, :dk, 0] = keys
    v = rng.standard_normal((1, T, 1, dv))
    q = np.zeros((1, T, 1, dk))
    q[0, -1, 0] = keys[3]
    x = dict(q=q, k=k, v=v, beta=np.ones((1, T, 1)), lam=np.zeros((1, T, 1)))
    o, c = O.recurrent(**x, variant=O.FALCON_1, eps=0.0)
    S = c["S"][0, 0]
    for j in range(dk):
        assert np.abs(keys[j] @ S - v[0, j + 1, 0]).max() <= 1e-12
    assert np.abs(o[0, -1, 0] - v[0, 4, 0]).max() <= 1e-12


# ---------------------------------------------------------------- P7
def test_p7_per_channel_with_equal_channels_is_scalar():
    rng = np.random.default_rng(15)
    x = rand_inputs(rng, 2, 26, 2, 6, 5)
    x2 = dict(x)
    x2["beta"] = np.repeat(x["beta"][..., None], 5, axis=-1)
    for v1, v2 in ((O.FALCON_1, O.FALCON_2), (O.FALCON_1A, O.FALCON_2A)):
        o1, c1 = O.recurrent(**x, variant=v1)
        o2, c2 = O.recurrent(**x2, variant=v2)
        assert np.abs(o1 - o2).max() <= 1e-14 and np.abs(c1["S"] - c2["S"]).max() <= 1e-14


def test_p7_per_channel_channels_are_independent_scalar_runs():
    """Each value channel of Falcon-2 is Falcon-1 on that channel alone with
    that channel's beta."""
    rng = np.random.default_rng(16)
    x = rand_inputs(rng, 1, 21, 1, 6, 4, per_channel=True)
    o2, c2 = O.recurrent(**x, variant=O.FALCON_2)
    for ch in range(4):
        xc = dict(q=x["q"], k=x["k"], v=x["v"][..., ch:ch + 1], beta=x["beta"][..., ch],
                  lam=x["lam"])
        o1, c1 = O.recurrent(**xc, variant=O.FALCON_1)
        assert np.abs(o1[..., 0] - o2[..., ch]).max() <= 1e-14
        assert np.abs(c1["S"][..., 0] - c2["S"][..., ch]).max() <= 1e-14


# ---------------------------------------------------------------- P8
@pytest.mark.parametrize("variant", ALL)
def test_p8_same_step_three_forms_agree(variant):
    rng = np.random.default_rng(300 + variant)
    W = 3 if O.is_windowed(variant) else 1
    x = rand_inputs(rng, 2, 45, 2, 8, 6, O.is_per_channel(variant))
    o_r, c_r = O.recurrent(**x, variant=variant, window=W, pairing="same")
    o_m, S_m = O.masked_parallel(**x, variant=variant, window=W, pairing="same")
    o_c, c_c = O.chunked(**x, variant=variant, window=W, chunk=16, pairing="same")
    assert rel(o_m, o_r) <= 1e-10 and rel(S_m, c_r["S"]) <= 1e-10
    assert rel(o_c, o_r) <= 1e-10 and rel(c_c["S"], c_r["S"]) <= 1e-10
    o_p, _ = O.recurrent(**x, variant=variant, window=W)
    assert rel(o_p, o_r) > 1e-3  # the two alignments are different methods


@pytest.mark.parametrize("variant", ALL)
def test_p8_same_step_is_prefix_alignment_of_the_next_key(variant):
    """Same-step pairs (k_t, v_t) are the prefix pairs of the key sequence
    shifted by one, with k_0 as the carried key of a sequence that already
    consumed one token."""
    rng = np.random.default_rng(310 + variant)
    W = 4 if O.is_windowed(variant) else 1
    B, T, H, dk, dv = 2, 37, 2, 8, 6
    x = rand_inputs(rng, B, T, H, dk, dv, O.is_per_channel(variant))
    o_s, c_s = O.recurrent(**x, variant=variant, window=W, pairing="same")
    k_next = np.zeros_like(x["k"])
    k_next[:, :-1] = x["k"][:, 1:]
    carry = {"S": np.zeros((B, H, dk, dv)), "k_prev": x["k"][:, 0].copy(),
             "pos": np.ones((B, H), dtype=np.int64)}
    if W > 1:
        carry["win_x"] = np.zeros((B, H, W - 1, dk))
        carry["win_v"] = np.zeros((B, H, W - 1, dv))
    xp = dict(x, k=k_next)
    o_p, c_p = O.recurrent(**xp, variant=variant, window=W, carry=carry)
    assert rel(o_s, o_p) <= 1e-12 and rel(c_s["S"], c_p["S"]) <= 1e-12


def test_p8_same_step_unit_step_reads_back_the_written_value():
    """Classical delta rule: gamma = 1, beta = 1, eps = 0, unit keys and
    q_t = k_t: after the write of (k_t, v_t) the state returns v_t for k_t,
    for any (non-orthogonal) key sequence."""
    rng = np.random.default_rng(320)
    T, dk, dv = 25, 6, 4
    k = rng.standard_normal((1, T, 1, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((1, T, 1, dv))
    x = dict(q=k.copy(), k=k, v=v, beta=np.ones((1, T, 1)), lam=np.zeros((1, T, 1)))
    o, _ = O.recurrent(**x, variant=O.FALCON_1, eps=0.0, pairing="same")
    assert np.abs(o - v).max() <= 1e-12
    o_p, _ = O.recurrent(**x, variant=O.FALCON_1, eps=0.0)
    assert np.abs(o_p - v).max() > 1e-2  # prefix-aligned pairs do not do this
