"""The allocation-free chunk forward (falcon_chunk_fwd_noalloc).

Callers such as plugin hosts that hand a library only tensors and a stream,
or services that forbid allocations once serving, cannot pass the scratch
buffer falcon_chunk_fwd needs; this entry point keeps its scratch in a fixed
array of the library instead.  The test calls it through the C ABI twice in a
row (the second call reuses the array the first one left behind) and checks
each result against falcon_chunk_fwd with a caller-owned workspace.  This file
is collected last so a failure here leaves every other test already run.
"""

from __future__ import annotations

import pytest
import torch

from helpers import TOL, params_for, rel_err
from workloads import FALCON_1, FALCON_1A, Workload, make_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import chunked_delta_rule_gb300 as F
    return F


def test_noalloc_matches_workspace_entry_point_twice(F):
    cases = [Workload("noalloc_f1", FALCON_1, 2, 300, 3, 64, 64, seed=61),
             Workload("noalloc_f1a", FALCON_1A, 1, 517, 2, 128, 128, seed=62)]
    for w in cases:  # two calls in a row on the shared scratch
        x = make_inputs(w, device="cuda")
        p = params_for(F, w)
        o_ref, c_ref = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
        o = torch.empty_like(o_ref)
        c = F.empty_carry(p)
        F.falcon_chunk_fwd_noalloc(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, c)
        torch.cuda.synchronize()
        assert rel_err(o.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= TOL["bf16"]
        assert rel_err(c["S"].cpu().numpy(), c_ref["S"].cpu().numpy()) <= TOL["bf16"]
        assert torch.equal(c["pos"], c_ref["pos"]) and torch.equal(c["k_prev"], c_ref["k_prev"])


def test_noalloc_rejects_what_it_cannot_cover(F):
    """Sizes beyond the fixed array and shapes outside the covered path are
    refused on the host, before anything is enqueued.  The too-big cases pass
    no tensors at all: if the size check ever moved after the launch, the
    call would stop at falcon_chunk_fwd's null-pointer check (INVALID_ARG)
    instead of touching memory."""
    big = [Workload("noalloc_big_d64", FALCON_1, 64, 4096, 16, 64, 64),     # 65536 chunks > 1927
           Workload("noalloc_big_d128", FALCON_1A, 1, 993 * 64, 1, 128, 128)]  # 993 chunks > 992
    for w in big:
        with pytest.raises(F.FalconError) as e:
            F.falcon_chunk_fwd_noalloc(params_for(F, w), None, None, None, None, None, None, None, None)
        assert e.value.code == -3, w.name
    for variant in (2, 3, 4, 5):  # outside the Falcon-1 / 1A tensor-core path
        w2 = Workload("noalloc_other", variant, 1, 64, 1, 64, 64, window=4 if variant >= 4 else 1)
        x = make_inputs(w2, device="cuda")
        o = torch.empty_like(x["v"])
        with pytest.raises(F.FalconError) as e:
            F.falcon_chunk_fwd_noalloc(params_for(F, w2), x["q"], x["k"], x["v"], x["beta"], x["lam"],
                                       None, o, None)
        assert e.value.code == -2


def test_noalloc_covers_its_stated_limit_at_d128(F):
    """992 chunks at d = 128, the largest problem the array holds there, runs
    and gives exactly the result of the workspace entry point; its status
    reads back clear."""
    w = Workload("noalloc_edge_d128", FALCON_1, 1, 992 * 64, 1, 128, 128, seed=63)
    x = make_inputs(w, device="cuda")
    p = params_for(F, w)
    o_ref, c_ref = F.chunk_forward(p, x["q"], x["k"], x["v"], x["beta"], x["lam"])
    o = torch.empty_like(o_ref)
    c = F.empty_carry(p)
    F.falcon_chunk_fwd_noalloc(p, x["q"], x["k"], x["v"], x["beta"], x["lam"], None, o, c)
    assert F.falcon_workspace_status(None) == F.FALCON_OK
    assert torch.equal(o, o_ref) and torch.equal(c["S"], c_ref["S"])
