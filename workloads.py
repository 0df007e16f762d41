"""Seeded synthetic inputs for the Falcon fast-weight forward.

This module holds no arithmetic of the method: it only draws random numbers
with ``torch.Generator`` on the CPU and lays them out in the library's
layouts.  The oracle (tests) and the CUDA path (tests, bench, smoke) both
take their inputs from here.

Recipe (shapes and distributions of the 124-130M-parameter models the
Falcon pages train: 12 heads of dimension 64, sequences of 2k and more):

* q, k ~ N(0, 1), then L2-normalised per token in fp32 (the feature map phi
  is the caller's; the library never applies it), then cast to the dtype.
* v ~ N(0, 1), cast to the dtype.
* beta = sigmoid(N(0, 1)) in fp32, shape [B, T, H] (or [B, T, H, dv] when
  the step is per value channel).
* gamma = sigmoid(N(mu, sd)) in fp32 and lambda = 1 - gamma; optionally a
  fraction of (b, t, h) positions is forced to gamma = 0 (lambda = 1) to
  exercise the positive-decay clamp.  The clamp itself is applied inside the
  library, not here.

Draw order is fixed (q, k, v, beta, gamma, forced mask) so every consumer
gets identical tensors for a given seed.
"""

from __future__ import annotations

from dataclasses import dataclass, field, replace

import torch

FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A = range(6)


@dataclass(frozen=True)
class Workload:
    name: str
    variant: int
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int = 64
    window: int = 1
    dtype: str = "bf16"           # "bf16" or "f32"
    seed: int = 0
    gamma_mu: float = 3.0
    gamma_sd: float = 1.0
    force_zero_gamma: float = 0.0  # fraction of positions with gamma forced to 0
    eps: float = 1e-6
    eps_gamma: float = 1e-3
    pairing: str = "prefix"       # "prefix" (x_t = k_{t-1}) or "same" (x_t = k_t, the ablation)

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)

    @property
    def per_channel(self) -> bool:
        return self.variant in (FALCON_2, FALCON_2A)


# The five workloads: one tiny check case and four layer shapes.
TINY_F1 = Workload("tiny_f1_1x64x1_d16", FALCON_1, 1, 64, 1, 16, 16, chunk=16,
                   dtype="f32", seed=0)
LM_F1A = Workload("lm124m_f1a_8x2048x12_d64", FALCON_1A, 8, 2048, 12, 64, 64, seed=1)
LM_F1 = LM_F1A.with_(name="lm124m_f1_8x2048x12_d64", variant=FALCON_1)
LONG_F1 = Workload("long_f1_2x16384x16_d128", FALCON_1, 2, 16384, 16, 128, 128, seed=2,
                   gamma_mu=4.0, gamma_sd=0.5, force_zero_gamma=0.01)
PERCH_F2 = Workload("perchannel_f2_4x4096x16_d128", FALCON_2, 4, 4096, 16, 128, 128, seed=3)
WINDOW_F3 = Workload("window_f3_4x8192x12_d64_w8", FALCON_3, 4, 8192, 12, 64, 64, window=8,
                     seed=4)
WINDOW_F3A = WINDOW_F3.with_(name="window_f3a_4x8192x12_d64_w8", variant=FALCON_3A)
WORKLOADS = [TINY_F1, LM_F1A, LM_F1, LONG_F1, PERCH_F2, WINDOW_F3, WINDOW_F3A]

# Decode: one token for 256 sequences x 12 heads, d = 64, fp32 state in HBM.
DECODE_B, DECODE_H, DECODE_D = 256, 12, 64


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    n = torch.sqrt((x * x).sum(-1, keepdim=True)).clamp_min(1e-12)
    return x / n


def make_inputs(w: Workload, seed: int | None = None, device="cpu") -> dict:
    """Draw one batch of inputs for workload ``w`` (CPU draw, then moved)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    shp_k = (w.B, w.T, w.H, w.dk)
    shp_v = (w.B, w.T, w.H, w.dv)
    q = _unit_rows(torch.randn(shp_k, generator=g)).to(dt)
    k = _unit_rows(torch.randn(shp_k, generator=g)).to(dt)
    v = torch.randn(shp_v, generator=g).to(dt)
    bshape = (w.B, w.T, w.H, w.dv) if w.per_channel else (w.B, w.T, w.H)
    beta = torch.sigmoid(torch.randn(bshape, generator=g))
    gamma = torch.sigmoid(w.gamma_mu + w.gamma_sd * torch.randn((w.B, w.T, w.H), generator=g))
    if w.force_zero_gamma > 0:
        mask = torch.rand((w.B, w.T, w.H), generator=g) < w.force_zero_gamma
        gamma = torch.where(mask, torch.zeros_like(gamma), gamma)
    lam = (1.0 - gamma).float()
    out = {"q": q, "k": k, "v": v, "beta": beta.float().contiguous(), "lam": lam.contiguous()}
    return {n: t.contiguous().to(device) for n, t in out.items()}


def make_carry(w: Workload, seed: int, pos: int | torch.Tensor, device="cpu",
               state_scale: float | None = None) -> dict:
    """A synthetic carry as if ``pos`` tokens were already consumed.

    S ~ N(0, 1/dk) (fp32), k_prev a unit feature, ring entries unit keys and
    N(0,1) values in the dtype.  Ring slots whose pair does not exist (global
    index < 1 with prefix alignment, < 0 with same-step pairing) are zero.
    """
    g = torch.Generator().manual_seed(seed)
    dt = torch_dtype(w.dtype)
    scale = (1.0 / w.dk) ** 0.5 if state_scale is None else state_scale
    S = torch.randn((w.B, w.H, w.dk, w.dv), generator=g) * scale
    k_prev = _unit_rows(torch.randn((w.B, w.H, w.dk), generator=g)).to(dt)
    if isinstance(pos, int):
        pos_t = torch.full((w.B, w.H), pos, dtype=torch.int64)
    else:
        pos_t = pos.to(torch.int64).reshape(w.B, w.H)
    out = {"S": S.float(), "k_prev": k_prev, "pos": pos_t}
    Wr = w.window - 1 if w.variant in (FALCON_3, FALCON_3A) else 0
    if Wr > 0:
        wx = _unit_rows(torch.randn((w.B, w.H, Wr, w.dk), generator=g)).to(dt)
        wv = torch.randn((w.B, w.H, Wr, w.dv), generator=g).to(dt)
        # zero slots that hold no pair: slot s holds the pair p in
        # [pos - Wr, pos - 1] with p mod Wr == s; it exists iff p >= first
        first = 0 if w.pairing == "same" else 1
        for b in range(w.B):
            for h in range(w.H):
                p0 = int(pos_t[b, h])
                for p in range(p0 - Wr, p0):
                    if p < first:
                        s = p % Wr
                        wx[b, h, s] = 0
                        wv[b, h, s] = 0
        out["win_x"] = wx
        out["win_v"] = wv
    if pos_t.min() == 0:
        zero = (pos_t == 0)
        out["k_prev"] = torch.where(zero[..., None], torch.zeros_like(k_prev), k_prev)
    return {n: t.contiguous().to(device) for n, t in out.items()}


def make_raw_inputs(w: Workload, seed: int | None = None, device="cpu") -> dict:
    """Raw projections and gate logits (for the library's prologue): q, k
    ~ N(0, s^2) with a per-token scale s ~ U(0.2, 5) (not normalised), v ~
    N(0, 1), beta logits ~ N(0, 1), lambda logits ~ N(-3, 1)."""
    g = torch.Generator().manual_seed(w.seed if seed is None else seed)
    dt = torch_dtype(w.dtype)
    shp_k = (w.B, w.T, w.H, w.dk)
    sq = 0.2 + 4.8 * torch.rand((w.B, w.T, w.H, 1), generator=g)
    sk = 0.2 + 4.8 * torch.rand((w.B, w.T, w.H, 1), generator=g)
    q = (torch.randn(shp_k, generator=g) * sq).to(dt)
    k = (torch.randn(shp_k, generator=g) * sk).to(dt)
    v = torch.randn((w.B, w.T, w.H, w.dv), generator=g).to(dt)
    bshape = (w.B, w.T, w.H, w.dv) if w.per_channel else (w.B, w.T, w.H)
    beta = torch.randn(bshape, generator=g)
    lam = -3.0 + torch.randn((w.B, w.T, w.H), generator=g)
    out = {"q": q, "k": k, "v": v, "beta": beta.float(), "lam": lam.float()}
    return {n: t.contiguous().to(device) for n, t in out.items()}


def pack_varlen(x: dict, lengths, device="cpu") -> tuple[dict, torch.Tensor]:
    """Pack batch rows b[:lengths[b]] of a [B, T, H, ...] input dict into
    [sum(lengths), H, ...] tensors; returns them and cu_seqlens (int32)."""
    packed = {n: torch.cat([t[b, :L] for b, L in enumerate(lengths)], dim=0).contiguous().to(device)
              for n, t in x.items()}
    cu = torch.tensor([0] + list(torch.cumsum(torch.tensor(lengths), 0).tolist()), dtype=torch.int32)
    return packed, cu.to(device)


def make_cotangents(w: Workload, seed: int, device="cpu", with_dS: bool = True) -> dict:
    """Cotangents for a backward pass: dO ~ N(0, 1) in the dtype (the shape
    of o) and dS_final ~ N(0, 1/dk) fp32 (or None)."""
    g = torch.Generator().manual_seed(seed)
    dO = torch.randn((w.B, w.T, w.H, w.dv), generator=g).to(torch_dtype(w.dtype))
    dS = torch.randn((w.B, w.H, w.dk, w.dv), generator=g) * (1.0 / w.dk) ** 0.5 if with_dS else None
    out = {"dO": dO, "dS_final": dS}
    return {n: (t.contiguous().to(device) if t is not None else None) for n, t in out.items()}


def make_decode_inputs(variant: int, window: int = 8, B: int = DECODE_B, H: int = DECODE_H,
                       d: int = DECODE_D, seed: int = 5, pos: int = 64, dtype: str = "bf16",
                       device="cpu") -> tuple[dict, dict, Workload]:
    """One decode token per sequence plus a carry at position ``pos`` (>= W)."""
    w = Workload(f"decode_{B}x{H}_d{d}", variant, B, 1, H, d, d, window=window, dtype=dtype,
                 seed=seed)
    inp = make_inputs(w, device=device)
    carry = make_carry(w, seed + 1000, pos, device=device)
    return inp, carry, w
