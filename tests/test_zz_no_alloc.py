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
    w = Workload("noalloc_big", FALCON_1, 64, 4096, 16, 64, 64)   # 64*16*64 chunks > 1927
    p = params_for(F, w)
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd_noalloc(p, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20, None, 1 << 20,
                                   None)
    assert e.value.code == -3
    for variant in (2, 3, 4, 5):  # outside the Falcon-1 / 1A tensor-core path
        w2 = Workload("noalloc_other", variant, 1, 64, 1, 64, 64, window=4 if variant >= 4 else 1)
        x = make_inputs(w2, device="cuda")
        o = torch.empty_like(x["v"])
        with pytest.raises(F.FalconError) as e:
            F.falcon_chunk_fwd_noalloc(params_for(F, w2), x["q"], x["k"], x["v"], x["beta"], x["lam"],
                                       None, o, None)
        assert e.value.code == -2
