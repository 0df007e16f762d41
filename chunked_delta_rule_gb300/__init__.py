"""Python binding of libfalcon.so (GB300 Falcon fast-weight forward).

Argument marshalling only: every step of the forward runs in the CUDA
kernels behind the C ABI declared in ``include/falcon.h``.  The functions
keep the C names; tensors are ``torch.Tensor`` on the GPU (their
``data_ptr()`` is passed) or raw integer device pointers.  There is no CPU
fallback: importing this package without a built ``libfalcon.so`` raises.
"""

from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libfalcon.so")

FALCON_1, FALCON_1A, FALCON_2, FALCON_2A, FALCON_3, FALCON_3A = range(6)
FALCON_BF16, FALCON_F32 = 0, 1
FALCON_IMPL_AUTO, FALCON_IMPL_GENERIC, FALCON_IMPL_TC, FALCON_IMPL_SCAN = 0, 1, 2, 3
FALCON_PAIR_PREFIX, FALCON_PAIR_SAME_STEP = 0, 1
FALCON_PROLOGUE_L2NORM_QK, FALCON_PROLOGUE_GATE_LOGITS = 1, 2
FALCON_OK = 0
FALCON_ERR_INVALID_ARG, FALCON_ERR_UNSUPPORTED, FALCON_ERR_WORKSPACE = -1, -2, -3
FALCON_ERR_CUDA, FALCON_ERR_TIMEOUT = -4, -5

EXPORTED = [
    "falcon_workspace_size", "falcon_chunk_fwd", "falcon_recurrent_step",
    "falcon_masked_parallel_workspace_size", "falcon_masked_parallel_ref_gpu",
    "falcon_strerror", "falcon_version", "falcon_chunk_fwd_plan", "falcon_chunk_fwd_timed",
    "falcon_chunk_fwd_noalloc", "falcon_backward_workspace_size", "falcon_backward",
    "falcon_backward_carry",
    "falcon_varlen_workspace_size", "falcon_chunk_fwd_varlen", "falcon_workspace_status",
    "falcon_test_hooks",
]


class FalconError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {strerror(code)} ({code})")


class falcon_params_t(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("T", ctypes.c_int32), ("H", ctypes.c_int32),
                ("dk", ctypes.c_int32), ("dv", ctypes.c_int32), ("chunk", ctypes.c_int32),
                ("window", ctypes.c_int32), ("eps", ctypes.c_float), ("eps_gamma", ctypes.c_float),
                ("variant", ctypes.c_int32), ("dtype", ctypes.c_int32), ("impl", ctypes.c_int32),
                ("pairing", ctypes.c_int32), ("prologue", ctypes.c_int32)]


class falcon_carry_t(ctypes.Structure):
    _fields_ = [("S", ctypes.c_void_p), ("k_prev", ctypes.c_void_p), ("win_x", ctypes.c_void_p),
                ("win_v", ctypes.c_void_p), ("pos", ctypes.c_void_p)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libfalcon.so once; raise if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    P, C, V, S = ctypes.POINTER(falcon_params_t), ctypes.POINTER(falcon_carry_t), ctypes.c_void_p, ctypes.c_size_t
    lib.falcon_workspace_size.argtypes = [P]
    lib.falcon_workspace_size.restype = S
    lib.falcon_chunk_fwd.argtypes = [P, V, V, V, V, V, C, V, C, V, S, V]
    lib.falcon_chunk_fwd.restype = ctypes.c_int
    lib.falcon_recurrent_step.argtypes = [P, V, V, V, V, V, C, V, V]
    lib.falcon_recurrent_step.restype = ctypes.c_int
    lib.falcon_masked_parallel_workspace_size.argtypes = [P]
    lib.falcon_masked_parallel_workspace_size.restype = S
    lib.falcon_masked_parallel_ref_gpu.argtypes = [P, V, V, V, V, V, V, V, V, S, V]
    lib.falcon_masked_parallel_ref_gpu.restype = ctypes.c_int
    lib.falcon_chunk_fwd_timed.argtypes = [P, V, V, V, V, V, C, V, C, V, S, V,
                                           ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32]
    lib.falcon_chunk_fwd_timed.restype = ctypes.c_int
    lib.falcon_chunk_fwd_noalloc.argtypes = [P, V, V, V, V, V, C, V, C, V]
    lib.falcon_chunk_fwd_noalloc.restype = ctypes.c_int
    lib.falcon_chunk_fwd_plan.argtypes = [P, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int32)]
    lib.falcon_chunk_fwd_plan.restype = ctypes.c_int
    lib.falcon_varlen_workspace_size.argtypes = [P]
    lib.falcon_varlen_workspace_size.restype = S
    lib.falcon_chunk_fwd_varlen.argtypes = [P, V, ctypes.c_int64, V, V, V, V, V, C, V, C, V, S, V]
    lib.falcon_chunk_fwd_varlen.restype = ctypes.c_int
    lib.falcon_backward_workspace_size.argtypes = [P]
    lib.falcon_backward_workspace_size.restype = S
    lib.falcon_backward.argtypes = [P, V, V, V, V, V, C, V, V, V, V, V, V, V, V, V, V, S, V]
    lib.falcon_backward.restype = ctypes.c_int
    lib.falcon_backward_carry.argtypes = [P, V, V, V, V, V, C, V, V, V, V, V, V, V, C, V, S, V]
    lib.falcon_backward_carry.restype = ctypes.c_int
    lib.falcon_workspace_status.argtypes = [V, V]
    lib.falcon_workspace_status.restype = ctypes.c_int
    lib.falcon_test_hooks.argtypes = [ctypes.c_uint64, ctypes.c_int32]
    lib.falcon_test_hooks.restype = None
    lib.falcon_strerror.argtypes = [ctypes.c_int]
    lib.falcon_strerror.restype = ctypes.c_char_p
    lib.falcon_version.argtypes = []
    lib.falcon_version.restype = ctypes.c_char_p
    _lib = lib
    return lib


@dataclass
class Params:
    """Python mirror of falcon_params_t."""
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int = 64
    window: int = 1
    eps: float = 1e-6
    eps_gamma: float = 1e-3
    variant: int = FALCON_1
    dtype: int = FALCON_BF16
    impl: int = FALCON_IMPL_AUTO
    pairing: int = FALCON_PAIR_PREFIX
    prologue: int = 0

    def c(self) -> falcon_params_t:
        return falcon_params_t(self.B, self.T, self.H, self.dk, self.dv, self.chunk, self.window,
                               self.eps, self.eps_gamma, self.variant, self.dtype, self.impl,
                               self.pairing, self.prologue)


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream
        except Exception:  # pragma: no cover
            return None
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def make_carry(carry: dict | None) -> falcon_carry_t | None:
    """Carry dict {S, k_prev, win_x, win_v, pos} -> falcon_carry_t (fields may be None)."""
    if carry is None:
        return None
    return falcon_carry_t(_ptr(carry.get("S")), _ptr(carry.get("k_prev")), _ptr(carry.get("win_x")),
                          _ptr(carry.get("win_v")), _ptr(carry.get("pos")))


def strerror(code: int) -> str:
    return load_library().falcon_strerror(code).decode()


def falcon_version() -> str:
    return load_library().falcon_version().decode()


def falcon_workspace_size(p: Params) -> int:
    return int(load_library().falcon_workspace_size(ctypes.byref(p.c())))


def falcon_masked_parallel_workspace_size(p: Params) -> int:
    return int(load_library().falcon_masked_parallel_workspace_size(ctypes.byref(p.c())))


def falcon_chunk_fwd_plan(p: Params) -> tuple[int, int]:
    """(impl, launches) the chunk forward uses for params p."""
    impl, n = ctypes.c_int32(0), ctypes.c_int32(0)
    _check(load_library().falcon_chunk_fwd_plan(ctypes.byref(p.c()), ctypes.byref(impl),
                                                 ctypes.byref(n)), "falcon_chunk_fwd_plan")
    return impl.value, n.value


def _check(code: int, where: str):
    if code != FALCON_OK:
        raise FalconError(code, where)


def falcon_chunk_fwd(p: Params, q, k, v, beta, lam, carry_in: dict | None, o,
                     carry_out: dict | None, workspace=None, workspace_bytes: int = 0, stream=None):
    lib = load_library()
    ci = make_carry(carry_in)
    co = make_carry(carry_out)
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    code = lib.falcon_chunk_fwd(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                                ctypes.byref(ci) if ci is not None else None, _ptr(o),
                                ctypes.byref(co) if co is not None else None, _ptr(workspace),
                                workspace_bytes, _stream(stream))
    _check(code, "falcon_chunk_fwd")


def falcon_chunk_fwd_timed(p: Params, q, k, v, beta, lam, carry_in: dict | None, o,
                           carry_out: dict | None, workspace, workspace_bytes: int, stream,
                           events: list):
    """falcon_chunk_fwd recording torch.cuda.Event objects around each kernel."""
    lib = load_library()
    ci = make_carry(carry_in)
    co = make_carry(carry_out)
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    code = lib.falcon_chunk_fwd_timed(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                      _ptr(lam), ctypes.byref(ci) if ci is not None else None,
                                      _ptr(o), ctypes.byref(co) if co is not None else None,
                                      _ptr(workspace), workspace_bytes, _stream(stream), arr,
                                      len(events))
    _check(code, "falcon_chunk_fwd_timed")


def falcon_chunk_fwd_noalloc(p: Params, q, k, v, beta, lam, carry_in: dict | None, o,
                             carry_out: dict | None, stream=None):
    """falcon_chunk_fwd without a workspace argument, for callers that cannot
    allocate device memory: the library uses its own fixed scratch array."""
    lib = load_library()
    ci = make_carry(carry_in)
    co = make_carry(carry_out)
    code = lib.falcon_chunk_fwd_noalloc(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                        _ptr(lam), ctypes.byref(ci) if ci is not None else None,
                                        _ptr(o), ctypes.byref(co) if co is not None else None,
                                        _stream(stream))
    _check(code, "falcon_chunk_fwd_noalloc")


def falcon_workspace_status(workspace=None, stream=None) -> int:
    """Status code of the last tensor-core call that used ``workspace`` (None:
    the last falcon_chunk_fwd_noalloc call on the current device): FALCON_OK
    or FALCON_ERR_TIMEOUT.  Synchronises the stream; clears the word."""
    code = load_library().falcon_workspace_status(_ptr(workspace), _stream(stream))
    if code not in (FALCON_OK, FALCON_ERR_TIMEOUT):
        _check(code, "falcon_workspace_status")
    return code


def falcon_test_hooks(wait_limit_ns: int = 0, stall: bool = False) -> None:
    """Failure-detection test hook: the bounded-wait limit of later calls
    (0 = the default 2 s) and a one-shot stall of the next Falcon-1/1A
    tensor-core call's per-chunk kernel."""
    load_library().falcon_test_hooks(int(wait_limit_ns), 1 if stall else 0)


def falcon_recurrent_step(p: Params, q, k, v, beta, lam, carry: dict, o, stream=None):
    lib = load_library()
    c = make_carry(carry)
    code = lib.falcon_recurrent_step(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(beta),
                                     _ptr(lam), ctypes.byref(c) if c is not None else None, _ptr(o),
                                     _stream(stream))
    _check(code, "falcon_recurrent_step")


def falcon_masked_parallel_ref_gpu(p: Params, q, k, v, beta, lam, o, S_final, workspace,
                                   workspace_bytes: int = 0, stream=None):
    lib = load_library()
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    code = lib.falcon_masked_parallel_ref_gpu(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v),
                                              _ptr(beta), _ptr(lam), _ptr(o), _ptr(S_final),
                                              _ptr(workspace), workspace_bytes, _stream(stream))
    _check(code, "falcon_masked_parallel_ref_gpu")


def falcon_varlen_workspace_size(p: Params) -> int:
    return int(load_library().falcon_varlen_workspace_size(ctypes.byref(p.c())))


def falcon_chunk_fwd_varlen(p: Params, cu_seqlens, total_tokens: int, q, k, v, beta, lam,
                            carry_in: dict | None, o, carry_out: dict | None, workspace,
                            workspace_bytes: int = 0, stream=None):
    lib = load_library()
    ci = make_carry(carry_in)
    co = make_carry(carry_out)
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    code = lib.falcon_chunk_fwd_varlen(ctypes.byref(p.c()), _ptr(cu_seqlens), int(total_tokens), _ptr(q),
                                       _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                                       ctypes.byref(ci) if ci is not None else None, _ptr(o),
                                       ctypes.byref(co) if co is not None else None, _ptr(workspace),
                                       workspace_bytes, _stream(stream))
    _check(code, "falcon_chunk_fwd_varlen")


def falcon_backward_workspace_size(p: Params) -> int:
    return int(load_library().falcon_backward_workspace_size(ctypes.byref(p.c())))


def falcon_backward(p: Params, q, k, v, beta, lam, carry_in: dict | None, dO, dS_final, dq, dk, dv,
                    dbeta, dlam, dS_in, dk_prev, workspace, workspace_bytes: int = 0, stream=None):
    lib = load_library()
    ci = make_carry(carry_in)
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    code = lib.falcon_backward(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                               ctypes.byref(ci) if ci is not None else None, _ptr(dO), _ptr(dS_final),
                               _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dlam), _ptr(dS_in),
                               _ptr(dk_prev), _ptr(workspace), workspace_bytes, _stream(stream))
    _check(code, "falcon_backward")


def falcon_backward_carry(p: Params, q, k, v, beta, lam, carry_in: dict | None, dO, dS_final, dq, dk, dv,
                          dbeta, dlam, dcarry: dict | None, workspace, workspace_bytes: int = 0, stream=None):
    """dcarry: dict of output buffers {S, k_prev, win_x, win_v} (any may be None)."""
    lib = load_library()
    ci = make_carry(carry_in)
    dc = make_carry(dcarry)
    if workspace is not None and not workspace_bytes and not isinstance(workspace, int):
        workspace_bytes = workspace.numel() * workspace.element_size()
    code = lib.falcon_backward_carry(ctypes.byref(p.c()), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(lam),
                                     ctypes.byref(ci) if ci is not None else None, _ptr(dO), _ptr(dS_final),
                                     _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbeta), _ptr(dlam),
                                     ctypes.byref(dc) if dc is not None else None, _ptr(workspace),
                                     workspace_bytes, _stream(stream))
    _check(code, "falcon_backward_carry")


# ---------------------------------------------------------------- tensor helpers
def alloc_workspace(nbytes: int, device="cuda"):
    """A 256-byte aligned byte buffer (torch's caching allocator aligns to 512)."""
    import torch
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def empty_carry(p: Params, device="cuda") -> dict:
    """Carry buffers for an output carry of params p."""
    import torch
    dt = torch.bfloat16 if p.dtype == FALCON_BF16 else torch.float32
    c = {"S": torch.empty((p.B, p.H, p.dk, p.dv), dtype=torch.float32, device=device),
         "k_prev": torch.empty((p.B, p.H, p.dk), dtype=dt, device=device),
         "pos": torch.empty((p.B, p.H), dtype=torch.int64, device=device)}
    if p.variant in (FALCON_3, FALCON_3A) and p.window > 1:
        c["win_x"] = torch.empty((p.B, p.H, p.window - 1, p.dk), dtype=dt, device=device)
        c["win_v"] = torch.empty((p.B, p.H, p.window - 1, p.dv), dtype=dt, device=device)
    return c


def chunk_forward(p: Params, q, k, v, beta, lam, carry_in: dict | None = None, want_carry=True,
                  stream=None):
    """Allocate o / carry_out / workspace with torch and call falcon_chunk_fwd."""
    import torch
    o = torch.empty((p.B, p.T, p.H, p.dv), dtype=q.dtype, device=q.device)
    co = empty_carry(p, q.device) if want_carry else None
    ws_n = falcon_workspace_size(p)
    ws = alloc_workspace(ws_n, q.device) if ws_n else None
    falcon_chunk_fwd(p, q, k, v, beta, lam, carry_in, o, co, ws, ws_n, stream)
    return o, co


def chunk_forward_varlen(p: Params, cu_seqlens, q, k, v, beta, lam, carry_in: dict | None = None,
                        want_carry=True, stream=None):
    """Packed sequences: q, k [total, H, dk], v [total, H, dv], cu_seqlens int32
    [B + 1] on the device; p.B = number of sequences, p.T >= the longest."""
    import torch
    total = q.shape[0]
    o = torch.empty((total, p.H, p.dv), dtype=q.dtype, device=q.device)
    co = empty_carry(p, q.device) if want_carry else None
    ws_n = falcon_varlen_workspace_size(p)
    ws = alloc_workspace(ws_n, q.device)
    falcon_chunk_fwd_varlen(p, cu_seqlens, total, q, k, v, beta, lam, carry_in, o, co, ws, ws_n, stream)
    return o, co


def masked_parallel(p: Params, q, k, v, beta, lam, stream=None):
    import torch
    o = torch.empty((p.B, p.T, p.H, p.dv), dtype=q.dtype, device=q.device)
    S = torch.empty((p.B, p.H, p.dk, p.dv), dtype=torch.float32, device=q.device)
    ws_n = falcon_masked_parallel_workspace_size(p)
    ws = alloc_workspace(ws_n, q.device)
    falcon_masked_parallel_ref_gpu(p, q, k, v, beta, lam, o, S, ws, ws_n, stream)
    return o, S



def backward(p: Params, q, k, v, beta, lam, dO, dS_final=None, carry_in: dict | None = None,
             stream=None) -> dict:
    """Allocate the gradients / workspace with torch and call falcon_backward_carry.

    Returns dq, dk, dv, dbeta, dlam, dS_in / dk_prev (gradients of the
    carried state and key) and, for Falcon-3/3A with W > 1, dwin_x / dwin_v
    (gradients of the carried window ring)."""
    import torch
    dev = q.device
    g = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
         "dbeta": torch.empty_like(beta), "dlam": torch.empty_like(lam),
         "dS_in": torch.empty((p.B, p.H, p.dk, p.dv), dtype=torch.float32, device=dev),
         "dk_prev": torch.empty((p.B, p.H, p.dk), dtype=q.dtype, device=dev)}
    dc = {"S": g["dS_in"], "k_prev": g["dk_prev"]}
    if p.variant in (FALCON_3, FALCON_3A) and p.window > 1:
        g["dwin_x"] = dc["win_x"] = torch.empty((p.B, p.H, p.window - 1, p.dk), dtype=q.dtype, device=dev)
        g["dwin_v"] = dc["win_v"] = torch.empty((p.B, p.H, p.window - 1, p.dv), dtype=q.dtype, device=dev)
    ws_n = falcon_backward_workspace_size(p)
    ws = alloc_workspace(ws_n, dev) if ws_n else None
    falcon_backward_carry(p, q, k, v, beta, lam, carry_in, dO, dS_final, g["dq"], g["dk"], g["dv"],
                          g["dbeta"], g["dlam"], dc, ws, ws_n, stream)
    return g


load_library()
