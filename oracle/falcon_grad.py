"""Gradients of the Falcon fast-weight forward: plain, slow, fp64 CPU
reference (the oracle of the backward pass).

TEST INFRASTRUCTURE ONLY, like the rest of this package: nothing in the
product path imports it, and it shares no code with the CUDA library.

The pages give no gradient formulas; training in the chunked framework they
describe [FW 三种等价形式; JC 三种视角看同一个更新] needs the gradient of the
forward with respect to q, k, v, beta, lambda and the carry.  Here the
forward recurrence of every variant (the same definition as
:func:`oracle.recurrent`, written step by step with torch CPU float64
tensors, including Falcon-3/3A's window of pairs and its carried ring) is
differentiated by torch's reverse-mode autodiff, a library primitive.
``tests/test_oracle_grad_pins.py`` pins it to the numpy oracle's forward and
to central finite differences.

The decay clamp gamma = clamp(1 - lambda, eps_gamma, 1) passes the gradient
where eps_gamma <= 1 - lambda <= 1 and stops it outside (torch.clamp).
"""

from __future__ import annotations

import numpy as np
import torch

from .falcon import (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A, effective_window,
                     is_additive, is_per_channel)

ONE_PAIR = (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A)
ALL = ONE_PAIR + (FALCON_3, FALCON_3A)


def recurrent_torch(q, k, v, beta, lam, variant, eps=1e-6, eps_gamma=1e-3, S_in=None,
                    k_prev=None, pos=None, pairing="prefix", window=1, win_x=None, win_v=None):
    """Forward of every variant with torch float64 ops (differentiable).

    Tensors: q, k [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H] (or
    [B, T, H, dv] per channel); lam [B, T, H]; S_in [B, H, dk, dv] or None;
    k_prev [B, H, dk] or None; pos [B, H] int (tokens consumed) or None;
    win_x [B, H, W-1, dk] / win_v [B, H, W-1, dv] the carried window ring
    (Falcon-3/3A, W > 1; pair p < 0 of this call sits in slot (pos + p)
    mod (W-1)) or None.  Per step t the window holds the pairs
    p = t-W+1 .. t; a pair exists iff its global index pos + p is >= 1
    (prefix alignment) or >= 0 (same-step); n_t counts the existing ones,
    e_t is their mean squared key norm and eta_t = beta_t / (eps + e_t)
    (no step when n_t = 0):
        Z = gamma_t S,  S = Z + (1/n_t) sum_p x_p (eta_t (.) r_p)^T,
        r_p = v_p - Z^T x_p (regression) or v_p (additive),  o_t = S^T q_t.
    Returns o [B, T, H, dv] and S_final [B, H, dk, dv].
    """
    assert variant in ALL
    W = effective_window(variant, window)
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    shift = 1 if pairing == "prefix" else 0
    S = torch.zeros((B, H, dk, dv), dtype=torch.float64) if S_in is None else S_in
    pos_t = torch.zeros((B, H), dtype=torch.int64) if pos is None else torch.as_tensor(pos)
    kp = torch.zeros((B, H, dk), dtype=torch.float64) if k_prev is None else k_prev
    gamma = torch.clamp(1.0 - lam, eps_gamma, 1.0)  # [B, T, H]
    per_ch = is_per_channel(variant)
    bi = torch.arange(B)[:, None]
    hi = torch.arange(H)[None, :]

    def pair(p):  # (x_p, v_p, exists) of local pair index p, as [B, H, .] tensors
        exists = ((pos_t + p) >= shift).to(torch.float64)
        if p >= 0:
            if shift == 0:
                x = k[:, p]
            else:
                x = kp if p == 0 else k[:, p - 1]
            return x, v[:, p], exists
        slot = torch.remainder(pos_t + p, W - 1)
        if win_x is None:  # no ring: such a pair must not exist
            z = torch.zeros((B, H), dtype=torch.float64)
            return (z[..., None].expand(B, H, dk), z[..., None].expand(B, H, dv), exists)
        return win_x[bi, hi, slot], win_v[bi, hi, slot], exists

    pairs = {p: pair(p) for p in range(-(W - 1), T)}
    outs = []
    for t in range(T):
        xs = torch.stack([pairs[p][0] for p in range(t - W + 1, t + 1)], dim=2)   # [B, H, W, dk]
        vs = torch.stack([pairs[p][1] for p in range(t - W + 1, t + 1)], dim=2)   # [B, H, W, dv]
        m = torch.stack([pairs[p][2] for p in range(t - W + 1, t + 1)], dim=2)    # [B, H, W]
        n = m.sum(-1)
        e = ((xs * xs).sum(-1) * m).sum(-1) / torch.clamp(n, min=1.0)
        has = (n > 0).to(torch.float64)
        denom = torch.where(n > 0, eps + e, torch.ones_like(e))
        if per_ch:
            eta = beta[:, t] / denom[..., None] * has[..., None]                       # [B, H, dv]
            coef = (m / torch.clamp(n, min=1.0)[..., None])[..., None] * eta[:, :, None, :]
        else:
            eta = beta[:, t] / denom * has                                              # [B, H]
            coef = (m * (eta / torch.clamp(n, min=1.0))[..., None])[..., None]          # [B, H, W, 1]
        Z = gamma[:, t][..., None, None] * S
        if is_additive(variant):
            r = vs
        else:
            r = vs - torch.einsum("bhwk,bhkv->bhwv", xs, Z)
        S = Z + torch.einsum("bhwk,bhwv->bhkv", xs, coef * r)
        outs.append(torch.einsum("bhk,bhkv->bhv", q[:, t], S))
    o = torch.stack(outs, dim=1) if T > 0 else torch.zeros((B, 0, H, dv), dtype=torch.float64)
    return o, S


def recurrent_vjp(q, k, v, beta, lam, variant, do, dS_final=None, eps=1e-6, eps_gamma=1e-3,
                  carry=None, pairing="prefix", window=1):
    """Gradient of L = <o, do> + <S_final, dS_final> with respect to every
    input of the forward (numpy in, numpy out, float64).

    carry: dict with S, k_prev, pos, win_x, win_v (any may be missing).
    Returns a dict with dq, dk, dv, dbeta, dlam, and dS_in / dk_prev /
    dwin_x / dwin_v for the carry fields supplied, plus the forward's o and S.
    """
    as_t = lambda a: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)
    tq, tk, tv, tb, tl = (as_t(a) for a in (q, k, v, beta, lam))
    S_in = kp = pos = wx = wv = None
    if carry is not None:
        if carry.get("S") is not None:
            S_in = as_t(carry["S"])
        if carry.get("k_prev") is not None:
            kp = as_t(carry["k_prev"])
        if carry.get("pos") is not None:
            pos = torch.as_tensor(np.asarray(carry["pos"], dtype=np.int64))
        if carry.get("win_x") is not None and effective_window(variant, window) > 1:
            wx = as_t(carry["win_x"])
            wv = as_t(carry["win_v"])
    o, S = recurrent_torch(tq, tk, tv, tb, tl, variant, eps, eps_gamma, S_in, kp, pos, pairing,
                           window, wx, wv)
    loss = (o * torch.as_tensor(np.asarray(do, dtype=np.float64))).sum()
    if dS_final is not None:
        loss = loss + (S * torch.as_tensor(np.asarray(dS_final, dtype=np.float64))).sum()
    named = [("dq", tq), ("dk", tk), ("dv", tv), ("dbeta", tb), ("dlam", tl), ("dS_in", S_in),
             ("dk_prev", kp), ("dwin_x", wx), ("dwin_v", wv)]
    named = [(n, x) for n, x in named if x is not None]
    grads = torch.autograd.grad(loss, [x for _, x in named], allow_unused=True)
    out = {n: (np.zeros(tuple(x.shape)) if gr is None else gr.numpy()) for (n, x), gr in zip(named, grads)}
    out["o"] = o.detach().numpy()
    out["S"] = S.detach().numpy()
    return out
