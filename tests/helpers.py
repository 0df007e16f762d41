"""Shared test helpers: run the GPU path through the C ABI and the oracle on
the same seeded inputs, and compare them."""

from __future__ import annotations

import numpy as np
import torch

import oracle

TOL = {"bf16": 2e-2, "f32": 1e-4}


def rel_err(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.abs(a - b).max() / max(np.abs(b).max(), 1e-30))


def to_np(d: dict | None) -> dict | None:
    if d is None:
        return None
    out = {}
    for k, v in d.items():
        if v is None:
            out[k] = None
        elif v.dtype == torch.int64:
            out[k] = v.detach().cpu().numpy()
        else:
            out[k] = v.detach().cpu().double().numpy()
    return out


def params_for(F, w, T=None, impl=None):
    return F.Params(B=w.B, T=w.T if T is None else T, H=w.H, dk=w.dk, dv=w.dv, chunk=w.chunk,
                    window=w.window, eps=w.eps, eps_gamma=w.eps_gamma, variant=w.variant,
                    dtype=F.FALCON_BF16 if w.dtype == "bf16" else F.FALCON_F32,
                    impl=F.FALCON_IMPL_AUTO if impl is None else impl,
                    pairing=F.FALCON_PAIR_SAME_STEP if w.pairing == "same" else F.FALCON_PAIR_PREFIX)


def oracle_full(w, x: dict, carry=None):
    xn = to_np(x)
    return oracle.recurrent(xn["q"], xn["k"], xn["v"], xn["beta"], xn["lam"], w.variant,
                            w.window, w.eps, w.eps_gamma, carry=to_np(carry), pairing=w.pairing)
