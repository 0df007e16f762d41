"""Gradients of the Falcon fast-weight forward: plain, slow, fp64 CPU
reference (the oracle of the backward pass).

TEST INFRASTRUCTURE ONLY, like the rest of this package: nothing in the
product path imports it, and it shares no code with the CUDA library.

The pages give no gradient formulas; training in the chunked framework they
describe [FW 三种等价形式; JC 三种视角看同一个更新] needs the gradient of the
forward with respect to q, k, v, beta, lambda and the carried state.  Here
the forward recurrence of the one-pair variants (Falcon-1, 1A, 2, 2A; the
same definition as :func:`oracle.recurrent`, written step by step with torch
CPU float64 tensors) is differentiated by torch's reverse-mode autodiff, a
library primitive.  ``tests/test_oracle_grad_pins.py`` pins it to the numpy
oracle's forward and to central finite differences.

The decay clamp gamma = clamp(1 - lambda, eps_gamma, 1) passes the gradient
where eps_gamma <= 1 - lambda <= 1 and stops it outside (torch.clamp).
"""

from __future__ import annotations

import numpy as np
import torch

from .falcon import FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, is_additive, is_per_channel

ONE_PAIR = (FALCON_1, FALCON_1A, FALCON_2, FALCON_2A)


def recurrent_torch(q, k, v, beta, lam, variant, eps=1e-6, eps_gamma=1e-3, S_in=None,
                    k_prev=None, pos=None, pairing="prefix"):
    """Forward of the one-pair variants with torch float64 ops (differentiable).

    Tensors: q, k [B, T, H, dk]; v [B, T, H, dv]; beta [B, T, H] (or
    [B, T, H, dv] per channel); lam [B, T, H]; S_in [B, H, dk, dv] or None;
    k_prev [B, H, dk] or None; pos [B, H] int (tokens consumed) or None.
    Returns o [B, T, H, dv] and S_final [B, H, dk, dv].
    """
    assert variant in ONE_PAIR
    B, T, H, dk = k.shape
    dv = v.shape[-1]
    shift = 1 if pairing == "prefix" else 0
    S = torch.zeros((B, H, dk, dv), dtype=torch.float64) if S_in is None else S_in
    pos_t = torch.zeros((B, H), dtype=torch.int64) if pos is None else torch.as_tensor(pos)
    kp = torch.zeros((B, H, dk), dtype=torch.float64) if k_prev is None else k_prev
    gamma = torch.clamp(1.0 - lam, eps_gamma, 1.0)  # [B, T, H]
    per_ch = is_per_channel(variant)
    outs = []
    for t in range(T):
        if shift == 1:
            x = kp if t == 0 else k[:, t - 1]           # [B, H, dk]
        else:
            x = k[:, t]
        exists = ((pos_t + t) >= shift).to(torch.float64)  # [B, H]
        n = (x * x).sum(-1)                            # [B, H]
        if per_ch:
            eta = beta[:, t] / (eps + n)[..., None] * exists[..., None]    # [B, H, dv]
        else:
            eta = (beta[:, t] / (eps + n) * exists)[..., None]             # [B, H, 1]
        Z = gamma[:, t][..., None, None] * S
        if is_additive(variant):
            delta = eta * v[:, t]
        else:
            r = v[:, t] - torch.einsum("bhk,bhkv->bhv", x, Z)
            delta = eta * r
        S = Z + x[..., :, None] * delta[..., None, :]
        outs.append(torch.einsum("bhk,bhkv->bhv", q[:, t], S))
    o = torch.stack(outs, dim=1) if T > 0 else torch.zeros((B, 0, H, dv), dtype=torch.float64)
    return o, S


def recurrent_vjp(q, k, v, beta, lam, variant, do, dS_final=None, eps=1e-6, eps_gamma=1e-3,
                  carry=None, pairing="prefix"):
    """Gradient of L = <o, do> + <S_final, dS_final> with respect to every
    input of the forward (numpy in, numpy out, float64).

    carry: dict with S, k_prev, pos (any may be missing).  Returns a dict with
    dq, dk, dv, dbeta, dlam, and dS_in / dk_prev when the carry supplies them.
    """
    as_t = lambda a: torch.tensor(np.asarray(a, dtype=np.float64), requires_grad=True)
    tq, tk, tv, tb, tl = (as_t(a) for a in (q, k, v, beta, lam))
    S_in = kp = pos = None
    if carry is not None:
        if carry.get("S") is not None:
            S_in = as_t(carry["S"])
        if carry.get("k_prev") is not None:
            kp = as_t(carry["k_prev"])
        if carry.get("pos") is not None:
            pos = torch.as_tensor(np.asarray(carry["pos"], dtype=np.int64))
    o, S = recurrent_torch(tq, tk, tv, tb, tl, variant, eps, eps_gamma, S_in, kp, pos, pairing)
    loss = (o * torch.as_tensor(np.asarray(do, dtype=np.float64))).sum()
    if dS_final is not None:
        loss = loss + (S * torch.as_tensor(np.asarray(dS_final, dtype=np.float64))).sum()
    leaves = [tq, tk, tv, tb, tl] + [x for x in (S_in, kp) if x is not None]
    grads = torch.autograd.grad(loss, leaves, allow_unused=True)
    g = [np.zeros(tuple(x.shape)) if gr is None else gr.numpy() for x, gr in zip(leaves, grads)]
    out = {"dq": g[0], "dk": g[1], "dv": g[2], "dbeta": g[3], "dlam": g[4]}
    i = 5
    if S_in is not None:
        out["dS_in"] = g[i]
        i += 1
    if kp is not None:
        out["dk_prev"] = g[i]
    out["o"] = o.detach().numpy()
    out["S"] = S.detach().numpy()
    return out
