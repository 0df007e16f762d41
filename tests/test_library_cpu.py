"""Host-side checks that need no GPU: the C-ABI library builds, loads and
exports every symbol include/falcon.h declares; argument errors are caught
on the host before anything is enqueued; workspace sizing."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def F():
    import __graft_entry__
    __graft_entry__.build()
    import chunked_delta_rule_gb300 as F
    return F


def declared_symbols():
    src = open(os.path.join(ROOT, "include", "falcon.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(falcon_[a-z_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(F):
    syms = declared_symbols()
    assert "falcon_chunk_fwd" in syms and "falcon_recurrent_step" in syms
    assert "falcon_masked_parallel_ref_gpu" in syms
    lib = ctypes.CDLL(F.LIB_PATH)
    for s in syms:
        assert hasattr(lib, s), s
    assert sorted(F.EXPORTED) == sorted(syms)


def test_version_and_strerror(F):
    assert "sm_103a" in F.falcon_version()
    for code in (0, -1, -2, -3, -4, -5):
        assert F.strerror(code)
    assert F.strerror(-99) == "unknown error"


def _p(F, **kw):
    base = dict(B=2, T=100, H=3, dk=64, dv=64, chunk=64, window=1, variant=F.FALCON_1,
                dtype=F.FALCON_BF16)
    base.update(kw)
    return F.Params(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(dk=48), -2), (dict(dv=256), -2), (dict(chunk=48), -2),
    (dict(variant=9), -1), (dict(dtype=7), -1), (dict(B=0), -1), (dict(T=-1), -1),
    (dict(eps=0.0), -1), (dict(eps_gamma=0.0), -1), (dict(eps_gamma=1.5), -1),
    (dict(variant=4, window=0), -2), (dict(variant=4, window=65), -2), (dict(impl=4), -1),
    (dict(impl=3), -2),
])
def test_chunk_fwd_rejects_bad_params_on_host(F, kw, code):
    p = _p(F, **kw)
    fake = 1 << 20  # never dereferenced: the call must return before enqueueing
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd(p, fake, fake, fake, fake, fake, None, fake, None, None, 0, 0)
    assert e.value.code == code


def test_null_pointers_rejected(F):
    p = _p(F)
    fake = 1 << 20
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd(p, None, fake, fake, fake, fake, None, fake, None, None, 0, 0)
    assert e.value.code == -1
    with pytest.raises(F.FalconError) as e:  # recurrent step needs T == 1 and a carry
        F.falcon_recurrent_step(_p(F, T=1), fake, fake, fake, fake, fake, None, fake, 0)
    assert e.value.code == -1
    with pytest.raises(F.FalconError) as e:
        F.falcon_recurrent_step(_p(F, T=2), fake, fake, fake, fake, fake,
                                {"S": fake, "k_prev": fake, "pos": fake}, fake, 0)
    assert e.value.code == -1


def test_overlapping_carries_rejected(F):
    p = _p(F)
    fake = 1 << 20
    c = {"S": 1 << 24, "k_prev": 1 << 25, "pos": 1 << 26}
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd(p, fake, fake, fake, fake, fake, c, fake, c, None, 0, 0)
    assert e.value.code == -1


def test_masked_parallel_limits(F):
    fake = 1 << 20
    with pytest.raises(F.FalconError) as e:
        F.falcon_masked_parallel_ref_gpu(_p(F, T=2048), fake, fake, fake, fake, fake, fake, fake,
                                         fake, 1 << 30, 0)
    assert e.value.code == -2
    with pytest.raises(F.FalconError) as e:  # workspace too small
        F.falcon_masked_parallel_ref_gpu(_p(F, T=100), fake, fake, fake, fake, fake, fake, fake,
                                         1 << 12, 16, 0)
    assert e.value.code == -3
    assert F.falcon_masked_parallel_workspace_size(_p(F, T=100)) > 0


def test_workspace_size_is_deterministic(F):
    p = _p(F, B=8, T=2048, H=12)
    n1 = F.falcon_workspace_size(p)
    n2 = F.falcon_workspace_size(p)
    assert n1 == n2 and n1 % 256 == 0
    assert F.falcon_workspace_size(_p(F, dk=48)) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(variant=4, window=35, dk=128, dv=128), -2), (dict(variant=5, window=65), -2),
    (dict(dk=32, dv=64), -2), (dict(dk=16, dv=16), -2), (dict(variant=9), -1), (dict(T=-1), -1),
])
def test_backward_rejects_bad_params_on_host(F, kw, code):
    """Params the host refuses before anything reaches the device (the
    addresses handed in are never dereferenced)."""
    p = _p(F, **kw)
    fake = 1 << 20
    with pytest.raises(F.FalconError) as e:
        F.falcon_backward(p, fake, fake, fake, fake, fake, None, fake, None, 1 << 22, 1 << 23,
                          1 << 24, 1 << 25, 1 << 26, None, None, 1 << 30, 1 << 30, 0)
    assert e.value.code == code
    assert F.falcon_backward_workspace_size(p) == 0


@pytest.mark.parametrize("kw", [dict(variant=4, window=8), dict(variant=5, window=34, dk=128, dv=128),
                                dict(variant=4, window=64), dict(variant=1, dk=128, dv=128),
                                dict(variant=2, dk=128, dv=128), dict(variant=4, window=1, dk=32, dv=32)])
def test_backward_window_kernel_workspace(F, kw):
    """Falcon-3/3A and d = 128 take the window kernel: the states at every
    64th step plus one recomputed block of 65 states, then per step and
    16-column group the partial sums (W + 1 d-vectors and two scalars,
    padded to 4 floats), and four scalars per step; all fp32."""
    p = _p(F, **kw)
    d, W = p.dk, (p.window if p.variant in (4, 5) else 1)
    kp = (W * d + d + 2 + 3) // 4 * 4
    BH, T = 2 * 3, 100
    want = BH * (2 + 64 + 1) * d * d + BH * T * (d // 16) * kp + BH * T * 4
    assert F.falcon_backward_workspace_size(p) == want * 4


def test_backward_workspace_and_overlap_checks(F):
    p = _p(F, B=2, T=100, H=3)
    n = F.falcon_backward_workspace_size(p)
    # chunked form (Falcon-1, d = 64): the status block, then per chunk eight 64 x 64 fp32
    # matrices (the chain transition's bf16 images take one) and 8 gate rows
    assert n == 256 + 2 * 3 * 2 * (8 * 64 * 64 + 8 * 64) * 4
    # recurrent form (d = 32, or an empty call): states at every 64th step + one block
    assert F.falcon_backward_workspace_size(_p(F, dk=32, dv=32)) == 2 * 3 * (2 + 64) * 32 * 32 * 4
    assert F.falcon_backward_workspace_size(_p(F, T=0)) == 2 * 3 * 64 * 64 * 64 * 4
    fake = 1 << 20
    outs = [1 << 22, 1 << 23, 1 << 24, 1 << 25, 1 << 26]
    with pytest.raises(F.FalconError) as e:  # workspace too small
        F.falcon_backward(p, fake, fake, fake, fake, fake, None, fake, None, *outs, None, None,
                          1 << 30, n - 1, 0)
    assert e.value.code == -3
    with pytest.raises(F.FalconError) as e:  # dq on top of q
        F.falcon_backward(p, fake, 1 << 27, 1 << 28, 1 << 29, 1 << 21, None, 1 << 31, None, fake,
                          *outs[1:], None, None, 1 << 32, n, 0)
    assert e.value.code == -1
    with pytest.raises(F.FalconError) as e:  # two gradients overlap
        F.falcon_backward(p, fake, 1 << 27, 1 << 28, 1 << 29, 1 << 21, None, 1 << 31, None,
                          1 << 22, 1 << 22, *outs[2:], None, None, 1 << 32, n, 0)
    assert e.value.code == -1
    with pytest.raises(F.FalconError) as e:  # null gradient with T > 0
        F.falcon_backward(p, fake, fake, fake, fake, fake, None, fake, None, None, *outs[1:], None,
                          None, 1 << 30, n, 0)
    assert e.value.code == -1


def test_prologue_and_varlen_sizes_and_flags(F):
    p = _p(F, B=3, T=200, H=2)
    base = F.falcon_workspace_size(p)
    p.prologue = 3
    with_pro = F.falcon_workspace_size(p)
    assert with_pro > base and with_pro % 256 == 0
    v = F.falcon_varlen_workspace_size(p)
    assert v > with_pro  # the padded outputs on top
    impl, n = F.falcon_chunk_fwd_plan(p)
    p.prologue = 0
    # bf16 Falcon-1 at d = 64 takes the prologue inside its two kernels; an
    # fp32 call (the portable path) applies it in one gather launch first
    assert n == F.falcon_chunk_fwd_plan(p)[1]
    q = _p(F, B=3, T=200, H=2, dtype=F.FALCON_F32)
    n0 = F.falcon_chunk_fwd_plan(q)[1]
    q.prologue = 3
    assert F.falcon_chunk_fwd_plan(q)[1] == n0 + 1
    p.prologue = 8
    assert F.falcon_workspace_size(p) == 0 and F.falcon_varlen_workspace_size(p) == 0
    fake = 1 << 20
    with pytest.raises(F.FalconError) as e:
        F.falcon_chunk_fwd(p, fake, fake, fake, fake, fake, None, fake, None, None, 0, 0)
    assert e.value.code == -1
    p.prologue = 1
    with pytest.raises(F.FalconError) as e:  # no cu_seqlens
        F.falcon_chunk_fwd_varlen(p, None, 10, fake, fake, fake, fake, fake, None, fake, None, fake, 1 << 30, 0)
    assert e.value.code == -1
    with pytest.raises(F.FalconError) as e:  # more tokens than B x T
        F.falcon_chunk_fwd_varlen(p, fake, 3 * 200 + 1, fake, fake, fake, fake, fake, None, fake, None, fake,
                                  1 << 30, 0)
    assert e.value.code == -1
    with pytest.raises(F.FalconError) as e:  # workspace too small
        F.falcon_chunk_fwd_varlen(p, fake, 10, fake, fake, fake, fake, fake, None, fake, None, 1 << 24, 16, 0)
    assert e.value.code == -3


@pytest.mark.parametrize("d", [64, 128])
def test_tc_workspace_layout(F, d):
    """Tensor-core forward workspace: a 256-byte status word, then per chunk
    the bf16 W | U images (2 d x 128 bytes) and a 1 KB gate slot, rounded up
    to 256 bytes (the layout the per-chunk and sequential kernels share)."""
    B, T, H = 2, 130, 3
    p = _p(F, B=B, T=T, H=H, dk=d, dv=d, impl=F.FALCON_IMPL_TC)
    nc = (T + 63) // 64
    want = 256 + B * H * nc * (2 * d * 128) + B * H * nc * 1024
    want = (want + 255) // 256 * 256
    assert F.falcon_workspace_size(p) == want


@pytest.mark.parametrize("kw,impl,launches", [
    # the tensor-core path: per-chunk kernel + sequential kernel (Falcon-1 / 1A)
    (dict(), "TC", 2), (dict(variant=1), "TC", 2), (dict(dk=128, dv=128), "TC", 2),
    # one tensor-core kernel each (Falcon-2 / 2A at d = 64 and 128)
    (dict(variant=2), "TC", 1), (dict(variant=3, dk=128, dv=128), "TC", 1),
    # Falcon-3A: per-chunk kernel + chain kernel
    (dict(variant=5, window=8), "TC", 2),
    # Falcon-3: per-chunk key-space kernel + chain kernel at d = 64 (W <= 9);
    # band prep + column-parallel window recurrence at d = 32
    (dict(variant=4, window=8), "TC", 2), (dict(variant=4, window=9), "TC", 2),
    (dict(variant=4, window=8, dk=32, dv=32), "SCAN", 2),
    # fp32 inputs, or a chunk other than 64: the portable chunk kernel
    (dict(dtype=1), "GENERIC", 1), (dict(chunk=32), "GENERIC", 1),
    # the prologue: inside the d = 64 Falcon-1 kernels, a gather launch elsewhere
    (dict(prologue=3), "TC", 2), (dict(prologue=3, variant=2), "TC", 2),
    (dict(prologue=1, dk=128, dv=128), "TC", 3),
])
def test_chunk_forward_plan(F, kw, impl, launches):
    """Which kernel family the AUTO plan picks and how many kernels it launches."""
    p = _p(F, **kw)
    got_impl, got_n = F.falcon_chunk_fwd_plan(p)
    assert got_impl == getattr(F, "FALCON_IMPL_" + impl) and got_n == launches
