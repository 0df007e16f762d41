"""Full-size parity of the two layer shapes whose own variant had no full-size
GPU case: Falcon-1 over 2 x 16384 x 16 heads at d = 128 (256 chunks per
head, 1 % of the decays forced to zero so the positive-decay floor binds,
[给记忆装一个“及时纠错”的开关, 数学上的稳定阀门:正衰减钳制]) and Falcon-1A over
8 x 2048 x 12 heads at d = 64.  Each runs in the launch configuration the
benchmark times (the default kernel family, caller workspace, carry out);
sampled heads are recomputed one by one by the oracle's token-by-token
recurrence, and the outputs and final states are compared element by
element.  The chunked form must equal the recurrence over the whole chain
[Falcon 家族重新对齐 fast-weight 记忆, 三种等价形式]."""

from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import TOL, params_for, rel_err
from workloads import LM_F1A, LONG_F1, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def _sampled_parity(F, w, heads, x):
    import oracle
    p = params_for(F, w)
    assert F.falcon_chunk_fwd_plan(p)[0] == F.FALCON_IMPL_TC
    o, co = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    torch.cuda.synchronize()
    assert torch.isfinite(o.float()).all() and torch.isfinite(co["S"]).all()
    sub = {}
    for key, val in x.items():
        sub[key] = np.stack([val[b, :, h].cpu().double().numpy() for b, h in heads])[:, :, None]
    errs = []
    for i, (b, h) in enumerate(heads):
        one = {key: val[i:i + 1] for key, val in sub.items()}
        o_ref, c_ref = oracle.recurrent(one["q"], one["k"], one["v"], one["beta"], one["lam"],
                                        w.variant, w.window, w.eps, w.eps_gamma)
        eo = rel_err(o[b, :, h].float().cpu().numpy(), o_ref[0, :, 0])
        eS = rel_err(co["S"][b, h].cpu().numpy(), c_ref["S"][0, 0])
        # the last 64 steps alone: the end of the chain, after every chunk
        eo_tail = rel_err(o[b, -64:, h].float().cpu().numpy(), o_ref[0, -64:, 0])
        errs.append((eo, eS, eo_tail))
        assert eo <= TOL["bf16"] and eS <= TOL["bf16"] and eo_tail <= TOL["bf16"], (b, h, errs[-1])
    assert co["pos"].eq(w.T).all()
    return errs


def test_long_context_d128_full_size_with_late_clamps(F):
    """2 x 16384 x 16 heads, d = 128: the state crosses 256 chunk boundaries,
    rounded to the MMA operand format at each one.  The sampled heads are
    chosen to have clamped (forced zero) decays in chunk 200 or later."""
    w = LONG_F1
    x = make_inputs(w, device="cuda")
    forced = (x["lam"] >= 1.0).cpu().numpy()   # lambda = 1: gamma = 0, floored at eps_gamma
    heads = []
    for b, h in [(0, 0), (1, 15), (0, 9), (1, 4)]:
        late = np.nonzero(forced[b, :, h])[0]
        late = late[late >= 200 * w.chunk]
        if late.size:
            heads.append((b, h))
    assert len(heads) >= 3, "the seeded draw has forced decays late in every sampled head"
    _sampled_parity(F, w, heads, x)


def test_lm124m_falcon1a_full_size(F):
    """Falcon-1A (additive write), 8 x 2048 x 12 heads, d = 64."""
    w = LM_F1A
    x = make_inputs(w, device="cuda")
    _sampled_parity(F, w, [(0, 0), (2, 5), (5, 9), (7, 11)], x)
