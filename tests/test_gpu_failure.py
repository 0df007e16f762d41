"""Failure detection of the tensor-core chunk forward (Falcon-1 at d = 64
and 128, Falcon-3 and Falcon-3A), tested without a GPU fault.  Every wait of those kernels is bounded; the test hook shortens the
limit and makes one wait, on a barrier that nothing completes, run out.  The
kernel must record the timeout in the workspace status word, give up its
chunks, free what it holds and return; the kernel after it must compute
nothing and write no carry; falcon_workspace_status must report
FALCON_ERR_TIMEOUT once (the read clears it); and the CUDA context must stay
usable, the next call giving the clean result.  No trap, fault or unbounded
wait is involved."""

from __future__ import annotations

import pytest
import torch

from helpers import TOL, oracle_full, params_for, rel_err
from workloads import LM_F1, LONG_F1, WINDOW_F3, WINDOW_F3A, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


@pytest.mark.parametrize("w", [LM_F1.with_(B=1, T=300, H=2), LONG_F1.with_(B=1, T=200, H=2,
                                                                             force_zero_gamma=0.0),
                               WINDOW_F3.with_(B=1, T=300, H=2), WINDOW_F3A.with_(B=1, T=300, H=2),
                               WINDOW_F3A.with_(B=1, T=1650, H=2)],
                         ids=["d64", "d128", "falcon3", "falcon3a", "falcon3a_groups"])
def test_stalled_wait_is_reported_and_the_context_survives(F, w):
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    impl, launches = F.falcon_chunk_fwd_plan(p)
    assert impl == F.FALCON_IMPL_TC
    if w.T == 1650:
        assert launches == 3   # Falcon-3A's chain in groups: the group-total kernel runs between
    n = F.falcon_workspace_size(p)
    ws = F.alloc_workspace(n)
    ws.fill_(0xFF)   # garbage in the status word: each call clears it when it starts

    def call(o, c):
        F.falcon_chunk_fwd(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, c, ws, n)

    o1 = torch.empty_like(x["v"])
    c1 = F.empty_carry(p)
    call(o1, c1)
    assert F.falcon_workspace_status(ws) == F.FALCON_OK
    o_ref, c_ref = oracle_full(w, x)
    assert rel_err(o1.float().cpu().numpy(), o_ref) <= TOL["bf16"]

    o2 = torch.zeros_like(x["v"])
    c2 = F.empty_carry(p)
    c2["pos"].fill_(-7)   # sentinel: a failed call writes no carry
    c2["S"].fill_(3.0)
    try:
        F.falcon_test_hooks(wait_limit_ns=2_000_000, stall=True)   # 2 ms
        call(o2, c2)
        assert F.falcon_workspace_status(ws) == F.FALCON_ERR_TIMEOUT
    finally:
        F.falcon_test_hooks(0, False)
    assert F.falcon_workspace_status(ws) == F.FALCON_OK   # the read cleared it
    assert bool((c2["pos"] == -7).all()) and bool((c2["S"] == 3.0).all())
    assert bool((o2 == 0).all()), "the sequential kernel skipped every chunk"

    o3 = torch.empty_like(x["v"])
    c3 = F.empty_carry(p)
    call(o3, c3)
    assert F.falcon_workspace_status(ws) == F.FALCON_OK
    assert torch.equal(o3, o1) and torch.equal(c3["S"], c1["S"]) and torch.equal(c3["pos"], c1["pos"])


def test_stall_hook_is_one_shot(F):
    """The stall applies to one call only; later calls run normally."""
    w = LM_F1.with_(B=1, T=130, H=1)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    n = F.falcon_workspace_size(p)
    ws = F.alloc_workspace(n)
    o = torch.empty_like(x["v"])
    try:
        F.falcon_test_hooks(wait_limit_ns=2_000_000, stall=True)
        for expect in (F.FALCON_ERR_TIMEOUT, F.FALCON_OK, F.FALCON_OK):
            F.falcon_chunk_fwd(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, None, ws, n)
            assert F.falcon_workspace_status(ws) == expect
    finally:
        F.falcon_test_hooks(0, False)
    o_ref, _ = oracle_full(w, x)
    assert rel_err(o.float().cpu().numpy(), o_ref) <= TOL["bf16"]
