"""Falcon fast-weight attention: plain, slow, fp64 CPU definitions (the oracle).

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports, calls or
links this module; only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It shares
no code with the CUDA library and imports nothing from it.

Sources (cited below by page title and section):

* [FW]   "把状态更新写成一条学习规则：Falcon 家族重新对齐 fast-weight 记忆"
         (zhouql-dev.github.io explainer of "Fast Weight Attention for
         Continual Learning").  Sections 本质, Falcon 家族, 三种等价形式.
* [JC]   "给记忆装一个“及时纠错”的开关：Falcon让循环模型学会边写边改"
         (long write-up).  Sections 一个被忽略的时间差, 把记忆更新变成一次梯度下降,
         Falcon家族六个变体各管一段, 数学上的稳定阀门:正衰减钳制,
         三种视角看同一个更新.
* [NEWS] chooseai.io news item on the same paper.  Section 核心方法.

The pages lost every formula in extraction, so the update is reconstructed
from their prose.  The readings taken where the prose is silent are listed
with the functions that rely on them:

* pair alignment: the state is written with the prefix-aligned pair
  (x_t, v_t) = (phi(k_{t-1}), v_t) [FW 本质; JC 一个被忽略的时间差].  phi is
  applied by the caller; x_0 is the carried previous key (zero when fresh).
  A pair whose global index is < 1 does not exist and writes nothing.
  The same-step pairing (x_t, v_t) = (phi(k_t), v_t), which the pages set
  against the prefix alignment as the usual delta-rule pairing
  [FW 本质; JC 一个被忽略的时间差], is available as an ablation
  (``pairing="same"``): every pair with global index >= 0 exists.
* shrink-then-correct: S_t = gamma_t S_{t-1} + eta_t x_t (v_t - gamma_t S_{t-1}^T x_t)^T,
  one online gradient step on the squared error at the shrunk state
  [JC 把记忆更新变成一次梯度下降], with the NLMS step
  eta_t = beta_t / (eps + ||x_t||^2) [JC same section; NEWS 核心方法] and the
  shrinkage lambda_t kept as its own knob [FW Falcon 家族; JC 这套框架真正解决的矛盾是什么].
* positive-decay clamp: gamma_t = 1 - lambda_t clamped to [eps_gamma, 1]
  [JC 数学上的稳定阀门:正衰减钳制].
* read after write: o_t = S_t^T q_t, no normaliser and no 1/sqrt(d)
  [FW 本质 and 三种等价形式 ("denominator-free")].
* Falcon-2: eta_t is a vector over the value channels [FW Falcon 家族;
  JC Falcon家族六个变体各管一段].
* Falcon-3: a mini-batch step over the last W existing pairs, with the
  statistics averaged over the window (not summed): the step uses the
  window-average energy e_t and the 1/n_t-averaged gradient [FW Falcon 家族;
  JC Falcon家族六个变体各管一段 and 写在后面].
* "A" variants: the inner-product objective makes the write purely additive,
  S_t = gamma_t S_{t-1} + eta_t x_t v_t^T (per channel / window-averaged for
  2A / 3A) [FW Falcon 家族; JC Falcon家族六个变体各管一段].

Every function works on numpy arrays in float64.  Layouts follow the C ABI:
q, k, v are [B, T, H, d]; beta is [B, T, H] (or [B, T, H, dv] for the
per-channel variants); lam is [B, T, H]; the carry holds S [B, H, dk, dv],
k_prev [B, H, dk], the window ring win_x [B, H, W-1, dk], win_v [B, H, W-1, dv]
and pos [B, H] (tokens already consumed).  Ring slot of the pair with global
index p is p mod (W-1); slots whose pair index is < 1 hold zeros.
"""

from __future__ import annotations

import numpy as np

FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A = range(6)
VARIANT_NAMES = {
    FALCON_1: "falcon1", FALCON_1A: "falcon1a", FALCON_2: "falcon2",
    FALCON_2A: "falcon2a", FALCON_3: "falcon3", FALCON_3A: "falcon3a",
}


def is_additive(variant: int) -> bool:
    """Inner-product ("A") objective: additive write [FW Falcon 家族]."""
    return variant in (FALCON_1A, FALCON_2A, FALCON_3A)


def is_per_channel(variant: int) -> bool:
    """Per-value-channel step eta_t in R^{dv} [JC Falcon家族六个变体各管一段]."""
    return variant in (FALCON_2, FALCON_2A)


def is_windowed(variant: int) -> bool:
    """Sliding-window mini-batch over the last W pairs [FW Falcon 家族]."""
    return variant in (FALCON_3, FALCON_3A)


def effective_window(variant: int, window: int) -> int:
    return int(window) if is_windowed(variant) else 1


def decay_factor(lam: np.ndarray, eps_gamma: float) -> np.ndarray:
    """gamma = 1 - lambda, kept >= eps_gamma so log(gamma) stays finite
    [JC 数学上的稳定阀门:正衰减钳制], and <= 1 (lambda is a shrinkage)."""
    return np.clip(1.0 - np.asarray(lam, dtype=np.float64), eps_gamma, 1.0)


def _f64(a):
    return None if a is None else np.asarray(a, dtype=np.float64)


PAIRINGS = ("prefix", "same")


def build_pairs(k, v, window, carry=None, pairing="prefix"):
    """Training pairs: prefix-aligned (x_j, v_j) = (k_{j-1}, v_j) [FW 本质], or
    same-step (k_j, v_j) for the ablation.

    Returns X [B, H, T+W-1, dk], V [B, H, T+W-1, dv] and valid [B, H, T+W-1]
    indexed by j + W - 1 for local pair index j in [-(W-1), T-1].  Prefix
    alignment: pair 0 uses the carried k_prev (zero when fresh) and a pair
    exists iff its global index pos + j is >= 1.  Same-step: pair j >= 0 uses
    k_j and exists iff pos + j >= 0.  Pairs j < 0 come from the carry's window
    ring in both.
    """
    assert pairing in PAIRINGS
    same = pairing == "same"
    k = _f64(k)
    v = _f64(v)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    W = int(window)
    L = T + W - 1
    X = np.zeros((B, H, L, dk))
    V = np.zeros((B, H, L, dv))
    kt = np.transpose(k, (0, 2, 1, 3))  # [B, H, T, dk]
    vt = np.transpose(v, (0, 2, 1, 3))
    pos = np.zeros((B, H), dtype=np.int64)
    if carry is not None:
        pos = np.asarray(carry["pos"], dtype=np.int64).reshape(B, H)
        if carry.get("k_prev") is not None and not same:
            X[:, :, W - 1, :] = _f64(carry["k_prev"])
    if same:
        X[:, :, W - 1:, :] = kt
    elif T > 1:
        X[:, :, W:, :] = kt[:, :, : T - 1, :]
    V[:, :, W - 1:, :] = vt
    if W > 1 and carry is not None and carry.get("win_x") is not None:
        wx = _f64(carry["win_x"])
        wv = _f64(carry["win_v"])
        for b in range(B):
            for h in range(H):
                for j in range(-(W - 1), 0):
                    slot = int((pos[b, h] + j) % (W - 1))
                    X[b, h, j + W - 1] = wx[b, h, slot]
                    V[b, h, j + W - 1] = wv[b, h, slot]
    j = np.arange(-(W - 1), T)
    valid = (pos[:, :, None] + j[None, None, :]) >= (0 if same else 1)
    X = X * valid[..., None]
    V = V * valid[..., None]
    return X, V, valid, pos


def step_coefficients(beta_t, x_win, valid_win, eps, per_channel):
    """NLMS step for one time step [JC 把记忆更新变成一次梯度下降; FW Falcon 家族].

    x_win [..., W, dk] / valid_win [..., W] are the pairs of the window.
    Returns the per-pair write coefficient eta_t / n_t (zero for missing pairs),
    shaped [..., W] or [..., W, dv] when eta is per channel.  n_t counts the
    existing pairs and e_t is their mean energy (window average).
    """
    n = valid_win.sum(axis=-1)
    energy = (x_win ** 2).sum(axis=-1) * valid_win
    e = energy.sum(axis=-1) / np.maximum(n, 1)
    has = n > 0                       # no existing pair: no step at all
    denom = np.where(has, eps + e, 1.0)
    if per_channel:
        eta = np.where(has[..., None], beta_t / denom[..., None], 0.0)  # [..., dv]
        coef = (valid_win / np.maximum(n, 1)[..., None])[..., None] * eta[..., None, :]
    else:
        eta = np.where(has, beta_t / denom, 0.0)
        coef = valid_win * (eta / np.maximum(n, 1))[..., None]
    return coef


def recurrent(q, k, v, beta, lam, variant, window=1, eps=1e-6, eps_gamma=1e-3,
              carry=None, return_trace=False, pairing="prefix"):
    """Token-by-token recurrence: the definition of every variant.

    The recurrent form is the inference form with an O(1) state per step
    [FW 三种等价形式; JC 三种视角看同一个更新].  Per step t, with the window
    W(t) of existing pairs among j in [t-W+1, t] (W = 1 outside Falcon-3),
    n_t = |W(t)|, e_t = mean_j ||x_j||^2 and eta_t = beta_t / (eps + e_t):

        Z_t = gamma_t S_{t-1}                              (shrinkage)
        regression:  S_t = Z_t + (1/n_t) sum_j x_j (eta_t * (v_j - Z_t^T x_j))^T
        additive:    S_t = Z_t + (1/n_t) sum_j x_j (eta_t * v_j)^T
        o_t = S_t^T q_t

    eta_t is a scalar (Falcon-1/1A/3/3A) or a dv-vector applied per channel
    (Falcon-2/2A).  With no existing pair the step only decays.

    Returns (o [B,T,H,dv], carry_out) and, with return_trace, a dict of
    per-step arrays: Z (shrunk state), S (state after the write),
    r (residual at the shrunk state for the newest pair), x, v, coef.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    beta = _f64(beta)
    lam = _f64(lam)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    W = effective_window(variant, window)
    per_ch = is_per_channel(variant)
    X, V, valid, pos = build_pairs(k, v, W, carry, pairing)
    S = np.zeros((B, H, dk, dv))
    if carry is not None and carry.get("S") is not None:
        S = _f64(carry["S"]).copy()
    gamma = decay_factor(lam, eps_gamma)  # [B, T, H]
    o = np.zeros((B, T, H, dv))
    trace = {"Z": [], "S": [], "r": [], "coef": []} if return_trace else None
    for t in range(T):
        xw = X[:, :, t:t + W, :]          # pairs j = t-W+1 .. t
        vw = V[:, :, t:t + W, :]
        mw = valid[:, :, t:t + W].astype(np.float64)
        g = gamma[:, t, :][:, :, None, None]
        Z = g * S
        coef = step_coefficients(beta[:, t, :], xw, mw, eps, per_ch)
        if is_additive(variant):
            resid = vw
        else:
            resid = vw - np.einsum("bhwk,bhkv->bhwv", xw, Z)
        if per_ch:
            delta = coef * resid           # [B, H, W, dv]
        else:
            delta = coef[..., None] * resid
        S = Z + np.einsum("bhwk,bhwv->bhkv", xw, delta)
        o[:, t, :, :] = np.einsum("bhk,bhkv->bhv", q[:, t, :, :], S)
        if return_trace:
            trace["Z"].append(Z)
            trace["S"].append(S.copy())
            trace["r"].append(vw[:, :, -1, :] - np.einsum("bhk,bhkv->bhv", xw[:, :, -1, :], Z))
            trace["coef"].append(coef)
    carry_out = make_carry_out(k, V, valid, X, S, pos, W, carry, T)
    if return_trace:
        return o, carry_out, trace
    return o, carry_out


def make_carry_out(k, V, valid, X, S, pos, W, carry, T):
    """State after the segment: S, last key, window ring and position."""
    B, _, H, dk = np.asarray(k).shape
    dv = V.shape[-1]
    k = _f64(k)
    if T >= 1:
        k_prev = np.transpose(k[:, T - 1:T, :, :], (0, 2, 1, 3))[:, :, 0, :].copy()
    elif carry is not None and carry.get("k_prev") is not None:
        k_prev = _f64(carry["k_prev"]).copy()
    else:
        k_prev = np.zeros((B, H, dk))
    out = {"S": S.copy(), "k_prev": k_prev, "pos": pos + T}
    if W > 1:
        wx = np.zeros((B, H, W - 1, dk))
        wv = np.zeros((B, H, W - 1, dv))
        for b in range(B):
            for h in range(H):
                for j in range(T - W + 1, T):
                    slot = int((pos[b, h] + j) % (W - 1))
                    idx = j + W - 1  # index into the pair arrays
                    if valid[b, h, idx]:
                        wx[b, h, slot] = X[b, h, idx]
                        wv[b, h, slot] = V[b, h, idx]
        out["win_x"] = wx
        out["win_v"] = wv
    return out


# --------------------------------------------------------------------------
# Masked-parallel form
# --------------------------------------------------------------------------

def masked_parallel(q, k, v, beta, lam, variant, window=1, eps=1e-6, eps_gamma=1e-3,
                    pairing="prefix"):
    """Masked-parallel form of a fresh sequence [FW 三种等价形式; JC 三种视角看同一个更新].

    The whole sequence is laid out at once, as in denominator-free linear
    attention (phi(Q) phi(K)^T (.) M) V: a lower-triangular decay mask
    M_ts = exp(g_t - g_s) (s <= t) built from the cumulative log-decay
    g_t = sum_{i<=t} log gamma_i over the full sequence, and, for the
    regression variants, a unit lower-triangular solve for the write
    residuals (the WY + TriSolve parallel view of Falcon-1 [FW 三种等价形式, 图4B]).

    Unknowns rho_{t,a} are the residuals of pair t-a at step t (a < W):
        rho_{t,a} = v_{t-a} - sum_{s<t} M_ts sum_b c_{s,b} (x_{t-a}.x_{s-b}) rho_{s,b}
    (regression; rho = v for the additive variants), where c_{s,b} is the
    write coefficient of pair s-b at step s.  Then
        o_t = sum_{s<=t} M_ts sum_b c_{s,b} (q_t . x_{s-b}) rho_{s,b}
        S_T = sum_s M_{T-1,s} sum_b c_{s,b} x_{s-b} rho_{s,b}^T.
    Per-channel steps give one such system per value channel.
    Returns (o [B,T,H,dv], S_final [B,H,dk,dv]).
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    beta = _f64(beta)
    lam = _f64(lam)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    W = effective_window(variant, window)
    per_ch = is_per_channel(variant)
    X, V, valid, _ = build_pairs(k, v, W, None, pairing)
    gamma = decay_factor(lam, eps_gamma)
    o = np.zeros((B, T, H, dv))
    S_final = np.zeros((B, H, dk, dv))
    for b in range(B):
        for h in range(H):
            g = np.cumsum(np.log(gamma[b, :, h]))
            M = np.tril(np.exp(np.minimum(g[:, None] - g[None, :], 0.0)))
            # coefficients c[s, a] (or [s, a, dv])
            coef = np.zeros((T, W, dv)) if per_ch else np.zeros((T, W))
            for s in range(T):
                xw = X[b, h, s:s + W]
                mw = valid[b, h, s:s + W].astype(np.float64)
                bt = beta[b, s, h]
                coef[s] = step_coefficients(bt, xw, mw, eps, per_ch)
            # unknown (t, a) is pair j = t - W + 1 + a (oldest first); its index
            # into the pair arrays is j + W - 1 = t + a
            pidx = np.array([[t + a for a in range(W)] for t in range(T)])
            Xu = X[b, h][pidx]            # [T, W, dk]
            Vu = V[b, h][pidx]            # [T, W, dv]
            G = np.einsum("tak,sbk->tasb", Xu, Xu)    # x_{t-a} . x_{s-b}
            P = np.einsum("tk,sbk->tsb", q[b, :, h, :], Xu)  # q_t . x_{s-b}
            strict = np.tril(np.ones((T, T)), -1)
            channels = range(dv) if per_ch else [None]
            rho = np.zeros((T, W, dv))
            for ch in channels:
                c = coef[..., ch] if per_ch else coef          # [T, W]
                rhs = Vu[..., ch] if per_ch else Vu             # [T, W] or [T, W, dv]
                if is_additive(variant):
                    sol = rhs
                else:
                    A = (M * strict)[:, None, :, None] * G * c[None, None, :, :]
                    A = A.reshape(T * W, T * W)
                    lhs = np.eye(T * W) + A
                    sol = np.linalg.solve(lhs, rhs.reshape(T * W, -1)).reshape(rhs.shape)
                if per_ch:
                    rho[..., ch] = sol
                else:
                    rho = sol
            cr = (coef * rho) if per_ch else (coef[..., None] * rho)   # [T, W, dv]
            o[b, :, h, :] = np.einsum("ts,tsb,sbv->tv", M, P, cr)
            S_final[b, h] = np.einsum("s,sbk,sbv->kv", M[T - 1], Xu, cr)
    return o, S_final


# --------------------------------------------------------------------------
# Chunked (SSD-style) form
# --------------------------------------------------------------------------

def chunked(q, k, v, beta, lam, variant, window=1, chunk=16, eps=1e-6, eps_gamma=1e-3,
            carry=None, pairing="prefix"):
    """Chunk-parallel form: cross-chunk state recurrence plus intra-chunk
    parallel work [FW 三种等价形式; JC 三种视角看同一个更新], with the per-chunk
    WY representation of the rank-one updates [FW 图4C; JC 三种视角看同一个更新].

    Per chunk with state S0 at its start, local cumulative log-decay
    g_r = sum_{i<=r} log gamma_i (inside the chunk) and Gamma_r = exp(g_r):

    Falcon-1 / 1A (one pair per step, scalar eta; pairs masked by existence):
        A_ri = eta_r exp(g_r - g_i) x_r.x_i   (i < r)       T = (I + A)^{-1}
        W = T diag(eta Gamma) X,  U = T diag(eta) V,  Delta = U - W S0
        (additive: Delta = diag(eta) V)
        O = diag(Gamma) Q S0 + (Q X^T (.) [exp(g_r - g_i)]_{i<=r}) Delta
        S1 = Gamma_last S0 + X^T diag(exp(g_last - g)) Delta
    Falcon-2 / 2A: one unit lower-triangular system per value channel,
        (I + diag(eta_.j) L) Delta_.j = eta_.j (V_.j - Gamma (X S0)_.j),
        L_ri = exp(g_r - g_i) x_r.x_i (i < r), solved for all channels with
        the shared L (the batched triangular solve [JC Falcon家族六个变体各管一段]).
    Falcon-3 / 3A: unknowns rho_{r,a} for the W pairs of every step, a
        (C W) x (C W) unit block-lower system built from the Gram matrix of the
        C + W - 1 distinct keys that the chunk's windows touch.
    Returns (o, carry_out) like :func:`recurrent`.
    """
    q = _f64(q)
    k = _f64(k)
    v = _f64(v)
    beta = _f64(beta)
    lam = _f64(lam)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    Wn = effective_window(variant, window)
    per_ch = is_per_channel(variant)
    X, V, valid, pos = build_pairs(k, v, Wn, carry, pairing)
    gamma = decay_factor(lam, eps_gamma)
    S = np.zeros((B, H, dk, dv))
    if carry is not None and carry.get("S") is not None:
        S = _f64(carry["S"]).copy()
    o = np.zeros((B, T, H, dv))
    for b in range(B):
        for h in range(H):
            S0 = S[b, h].copy()
            for c0 in range(0, T, chunk):
                c1 = min(c0 + chunk, T)
                C = c1 - c0
                g = np.cumsum(np.log(gamma[b, c0:c1, h]))
                Gam = np.exp(g)
                decay = np.exp(np.minimum(g[:, None] - g[None, :], 0.0))  # exp(g_r - g_i)
                Qc = q[b, c0:c1, h, :]
                coef = np.stack([
                    step_coefficients(beta[b, t, h], X[b, h, t:t + Wn],
                                      valid[b, h, t:t + Wn].astype(np.float64), eps, per_ch)
                    for t in range(c0, c1)])       # [C, Wn] or [C, Wn, dv]
                if Wn == 1 and not per_ch:
                    S0, Oc = _chunk_wy(Qc, X[b, h, c0:c1], V[b, h, c0:c1], coef[:, 0],
                                       g, Gam, decay, S0, variant)
                elif Wn == 1:
                    S0, Oc = _chunk_per_channel(Qc, X[b, h, c0:c1], V[b, h, c0:c1],
                                                coef[:, 0, :], g, Gam, decay, S0, variant)
                else:
                    S0, Oc = _chunk_window(Qc, X[b, h, c0:c1 + Wn - 1], V[b, h, c0:c1 + Wn - 1],
                                           coef, g, Gam, decay, S0, variant, Wn)
                o[b, c0:c1, h, :] = Oc
            S[b, h] = S0
    carry_out = make_carry_out(k, V, valid, X, S, pos, Wn, carry, T)
    return o, carry_out


def _chunk_wy(Q, X, V, eta, g, Gam, decay, S0, variant):
    """One Falcon-1/1A chunk in the WY form (T, W, U, Delta)."""
    C = X.shape[0]
    lower_incl = np.tril(np.ones((C, C)))
    if is_additive(variant):
        Delta = eta[:, None] * V
    else:
        G = X @ X.T
        A = eta[:, None] * decay * G * np.tril(np.ones((C, C)), -1)
        Tm = np.linalg.inv(np.eye(C) + A)
        Wm = Tm @ ((eta * Gam)[:, None] * X)
        U = Tm @ (eta[:, None] * V)
        Delta = U - Wm @ S0
    P = (Q @ X.T) * decay * lower_incl
    O = Gam[:, None] * (Q @ S0) + P @ Delta
    S1 = Gam[-1] * S0 + X.T @ (np.exp(g[-1] - g)[:, None] * Delta)
    return S1, O


def _chunk_per_channel(Q, X, V, eta, g, Gam, decay, S0, variant):
    """One Falcon-2/2A chunk: the row-scaled triangular solve shared by all
    value channels (L is common, eta differs per channel)."""
    C = X.shape[0]
    lower_incl = np.tril(np.ones((C, C)))
    if is_additive(variant):
        Delta = eta * V
    else:
        L = decay * (X @ X.T) * np.tril(np.ones((C, C)), -1)
        rhs = eta * (V - Gam[:, None] * (X @ S0))
        Delta = np.zeros_like(rhs)
        for r in range(C):  # forward substitution, all channels at once
            Delta[r] = rhs[r] - eta[r] * (L[r, :r] @ Delta[:r])
    P = (Q @ X.T) * decay * lower_incl
    O = Gam[:, None] * (Q @ S0) + P @ Delta
    S1 = Gam[-1] * S0 + X.T @ (np.exp(g[-1] - g)[:, None] * Delta)
    return S1, O


def _chunk_window(Q, Xk, Vk, coef, g, Gam, decay, S0, variant, Wn):
    """One Falcon-3/3A chunk.  Xk/Vk hold the C + W - 1 pairs touched by the
    chunk; slot a of step r (oldest first) is pair index r + a."""
    C = Q.shape[0]
    per_ch = coef.ndim == 3
    dv = Vk.shape[-1]
    pidx = np.array([[r + a for a in range(Wn)] for r in range(C)])
    Xu = Xk[pidx]                  # [C, W, dk]
    Vu = Vk[pidx]                  # [C, W, dv]
    Gk = Xk @ Xk.T                 # Gram of the distinct keys
    G = Gk[pidx][:, :, pidx]       # [C, W, C, W]
    if is_additive(variant):
        rho = Vu
    else:
        rhs = Vu - Gam[:, None, None] * np.einsum("rak,kv->rav", Xu, S0)
        strict = np.tril(np.ones((C, C)), -1) * decay
        if per_ch:
            rho = np.zeros_like(rhs)
            for ch in range(dv):
                A = strict[:, None, :, None] * G * coef[None, None, :, :, ch]
                lhs = np.eye(C * Wn) + A.reshape(C * Wn, C * Wn)
                rho[..., ch] = np.linalg.solve(lhs, rhs[..., ch].reshape(-1)).reshape(C, Wn)
        else:
            A = strict[:, None, :, None] * G * coef[None, None, :, :]
            lhs = np.eye(C * Wn) + A.reshape(C * Wn, C * Wn)
            rho = np.linalg.solve(lhs, rhs.reshape(C * Wn, dv)).reshape(C, Wn, dv)
    cr = coef * rho if per_ch else coef[..., None] * rho
    P = np.einsum("rk,sbk->rsb", Q, Xu)
    O = Gam[:, None] * (Q @ S0) + np.einsum("rs,rsb,sbv->rv", decay * np.tril(np.ones((C, C))), P, cr)
    S1 = Gam[-1] * S0 + np.einsum("s,sbk,sbv->kv", np.exp(g[-1] - g), Xu, cr)
    return S1, O


# --------------------------------------------------------------------------
# Helpers for parity at full size
# --------------------------------------------------------------------------

def recurrent_heads(q, k, v, beta, lam, variant, heads, window=1, eps=1e-6, eps_gamma=1e-3,
                    carry=None, pairing="prefix"):
    """Run :func:`recurrent` on a subset of (b, h) pairs only.

    heads: list of (b, h).  Returns o [len(heads), T, dv] and S_final
    [len(heads), dk, dv].  Each head is an independent recurrence, so this is
    the definition evaluated on fewer heads.
    """
    outs, states = [], []
    for (b, h) in heads:
        sub = lambda a: None if a is None else np.asarray(a)[b:b + 1, :, h:h + 1]
        c = None
        if carry is not None:
            c = {key: (None if val is None else np.asarray(val)[b:b + 1, h:h + 1])
                 for key, val in carry.items()}
        o, co = recurrent(sub(q), sub(k), sub(v), sub(beta), sub(lam), variant, window,
                          eps, eps_gamma, c, pairing=pairing)
        outs.append(o[0, :, 0, :])
        states.append(co["S"][0, 0])
    return np.stack(outs), np.stack(states)
