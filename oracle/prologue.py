"""The steps either side of the Falcon forward, plain fp64 numpy (oracle).

TEST INFRASTRUCTURE ONLY, like the rest of this package: nothing in the
product path imports it, and it shares no code with the CUDA library.

* Feature map phi [FW 三种等价形式 (phi(Q), phi(K) in the linear-attention
  form); JC 三种视角看同一个更新]: the pages leave phi open; the reading
  taken (and the one the synthetic workloads use) is the per-token L2
  normalisation phi(x) = x / max(|x|_2, 1e-12).
* Gates from logits [JC 把记忆更新变成一次梯度下降 (beta and lambda as
  learned knobs, each in (0, 1))]: beta = sigmoid(b), lambda = sigmoid(a),
  so the decay gamma = 1 - lambda = sigmoid(-a) before its eps_gamma floor.
* Packed sequences: each sequence of a packed batch is its own recurrence
  (its own carry); ``recurrent_varlen`` runs the definition on each one.
"""

from __future__ import annotations

import numpy as np

from .falcon import recurrent

L2NORM_QK, GATE_LOGITS = 1, 2


def phi(x):
    """Per-token L2 normalisation over the last axis, fp64."""
    x = np.asarray(x, dtype=np.float64)
    n = np.sqrt((x * x).sum(-1, keepdims=True))
    return x / np.maximum(n, 1e-12)


def sigmoid(x):
    """Logistic function, evaluated without cancellation on either side:
    1 / (1 + e^-x) for x >= 0, e^x / (1 + e^x) for x < 0."""
    x = np.asarray(x, dtype=np.float64)
    ex = np.exp(-np.abs(x))
    return np.where(x >= 0, 1.0 / (1.0 + ex), ex / (1.0 + ex))


def apply_prologue(q, k, beta, lam, flags):
    """Inputs as the forward consumes them (features, gates) from the raw
    ones, per the prologue flags."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    beta = np.asarray(beta, dtype=np.float64)
    lam = np.asarray(lam, dtype=np.float64)
    if flags & L2NORM_QK:
        q, k = phi(q), phi(k)
    if flags & GATE_LOGITS:
        beta, lam = sigmoid(beta), sigmoid(lam)
    return q, k, beta, lam


def recurrent_varlen(q, k, v, beta, lam, cu_seqlens, variant, window=1, eps=1e-6, eps_gamma=1e-3,
                     carries=None, pairing="prefix"):
    """Packed sequences [total, H, .] delimited by cu_seqlens: the recurrence
    of each sequence on its own.  carries: list (one dict or None per
    sequence, leading axes [1, H, ...]).  Returns the packed outputs and the
    list of per-sequence carries."""
    cu = [int(c) for c in np.asarray(cu_seqlens)]
    outs, cos = [], []
    for i in range(len(cu) - 1):
        s, e = cu[i], cu[i + 1]
        sl = lambda a: np.asarray(a, dtype=np.float64)[s:e][None]
        ci = None if carries is None else carries[i]
        if e == s:
            cos.append(ci)
            outs.append(np.zeros((0,) + np.asarray(v).shape[1:]))
            continue
        o, co = recurrent(sl(q), sl(k), sl(v), sl(beta), sl(lam), variant, window, eps, eps_gamma,
                          carry=ci, pairing=pairing)
        outs.append(o[0])
        cos.append(co)
    return np.concatenate(outs, axis=0), cos
