"""Pins of the prologue and varlen parts of the oracle (oracle/prologue.py):
the feature map against its invariants and a hand value, the sigmoid
against its exponential closed form and symmetry, and packed sequences
against separate runs of the definition."""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from workloads import FALCON_1, FALCON_2, FALCON_3, Workload, make_inputs, pack_varlen


def test_phi_invariants():
    rng = np.random.default_rng(3)
    x = rng.normal(size=(5, 7, 16)) * rng.uniform(0.1, 10, size=(5, 7, 1))
    y = oracle.phi(x)
    assert np.allclose(np.linalg.norm(y, axis=-1), 1.0, atol=1e-14)
    assert np.allclose(oracle.phi(3.5 * x), y, atol=1e-14)           # scale invariant
    assert np.allclose(oracle.phi([3.0, 4.0]), [0.6, 0.8], atol=1e-15)  # hand value
    assert np.all(oracle.phi(np.zeros(8)) == 0.0)                    # zero stays zero
    assert np.allclose((y * x).sum(-1), np.linalg.norm(x, axis=-1))  # same direction


def test_sigmoid_closed_form_and_symmetry():
    a = np.linspace(-30, 30, 121)
    assert np.allclose(oracle.sigmoid(a), 1.0 / (1.0 + np.exp(-a)), rtol=1e-14, atol=1e-300)
    assert np.allclose(oracle.sigmoid(a) + oracle.sigmoid(-a), 1.0, atol=1e-15)
    assert oracle.sigmoid(0.0) == 0.5


def test_apply_prologue_flags():
    w = Workload("p", FALCON_1, 1, 9, 2, 8, 8, dtype="f32", seed=4)
    x = {n: t.double().numpy() for n, t in make_inputs(w).items()}
    q, k, b, l = oracle.apply_prologue(x["q"], x["k"], x["beta"], x["lam"], 0)
    assert np.array_equal(q, x["q"]) and np.array_equal(l, x["lam"])
    q, k, b, l = oracle.apply_prologue(x["q"] * 7, x["k"] * 0.1, x["beta"], x["lam"], oracle.L2NORM_QK)
    assert np.allclose(q, x["q"] / np.linalg.norm(x["q"], axis=-1, keepdims=True))
    _, _, b, l = oracle.apply_prologue(x["q"], x["k"], np.zeros(3), np.array([-np.inf, 0.0, np.inf]),
                                       oracle.GATE_LOGITS)
    assert np.allclose(b, 0.5) and np.allclose(l, [0.0, 0.5, 1.0])  # lambda = 1: gamma floored


@pytest.mark.parametrize("variant,window", [(FALCON_1, 1), (FALCON_2, 1), (FALCON_3, 4)])
def test_varlen_is_separate_sequences(variant, window):
    w = Workload("v", variant, 4, 30, 2, 8, 8, window=window, dtype="f32", seed=5 + variant)
    x = {n: t.double() for n, t in make_inputs(w).items()}
    lengths = [30, 0, 1, 17]
    packed, cu = pack_varlen(x, lengths)
    pn = {n: t.numpy() for n, t in packed.items()}
    o, cos = oracle.recurrent_varlen(pn["q"], pn["k"], pn["v"], pn["beta"], pn["lam"], cu.numpy(),
                                     variant, window)
    assert o.shape[0] == sum(lengths)
    s = 0
    for b, L in enumerate(lengths):
        if L == 0:
            assert cos[b] is None
            continue
        xb = {n: t[b:b + 1, :L].numpy() for n, t in x.items()}
        ob, cb = oracle.recurrent(xb["q"], xb["k"], xb["v"], xb["beta"], xb["lam"], variant, window)
        assert np.array_equal(o[s:s + L], ob[0])
        assert np.array_equal(cos[b]["S"], cb["S"])
        s += L
    # order of the sequences does not matter
    perm = [3, 0, 2, 1]
    packed2, cu2 = pack_varlen({n: t[perm] for n, t in x.items()}, [lengths[i] for i in perm])
    p2 = {n: t.numpy() for n, t in packed2.items()}
    o2, _ = oracle.recurrent_varlen(p2["q"], p2["k"], p2["v"], p2["beta"], p2["lam"], cu2.numpy(),
                                    variant, window)
    assert np.array_equal(o2[:17], o[31:48])
