"""Thin Python binding of the Relation C ABI (include/relation.h).

The functions named like the C entry points (``relation_fwd``,
``relation_bwd``, ...) marshal torch CUDA tensors into pointers and call the
library; every step of the computation runs in the library's CUDA kernels.
PyTorch provides device memory and streams only.  There is no fallback: if the
library is missing or a call fails, an exception is raised.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

import torch

from . import build as _build

RELATION_F32 = 0
RELATION_BF16 = 1
RELATION_LAYOUT_BHTD = 0  # operands [B, H, T, d_h]
RELATION_LAYOUT_BTHD = 1  # operands [B, T, H, d_h]

STATUS = {
    0: "RELATION_OK",
    1: "RELATION_ERR_INVALID_ARGUMENT",
    2: "RELATION_ERR_UNSUPPORTED",
    3: "RELATION_ERR_MISALIGNED",
    4: "RELATION_ERR_WORKSPACE_TOO_SMALL",
    5: "RELATION_ERR_CUDA",
    6: "RELATION_ERR_DEVICE_TIMEOUT",
    7: "RELATION_ERR_DEVICE_UNSAFE",
}


class RelationError(RuntimeError):
    def __init__(self, code: int, what: str, message: str):
        super().__init__(f"{what}: {STATUS.get(code, code)} ({message})")
        self.code = code


class Problem(ctypes.Structure):
    """Mirror of relation_problem_t."""

    _fields_ = [
        ("B", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("T", ctypes.c_int64),
        ("d_h", ctypes.c_int64),
        ("dtype", ctypes.c_int32),
        ("tau_S", ctypes.c_float),
        ("lam", ctypes.c_float),
        ("causal", ctypes.c_int32),
        ("layout", ctypes.c_int32),
    ]


_lock = threading.Lock()
_lib = None

_VP = ctypes.c_void_p
_BWD_ARGTYPES = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = True) -> ctypes.CDLL:
    """Loads the in-tree library (building it first when missing or stale)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if build_if_missing and not _build.up_to_date():
            _build.build()
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"Relation CUDA library not built at {_build.LIB}")
        lib = ctypes.CDLL(_build.LIB)
        lib.relation_fwd.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP]
        lib.relation_fwd.restype = ctypes.c_int
        lib.relation_fwd_workspace_bytes.argtypes = [ctypes.POINTER(Problem)]
        lib.relation_fwd_workspace_bytes.restype = ctypes.c_size_t
        lib.relation_fwd_ws.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]
        lib.relation_fwd_ws.restype = ctypes.c_int
        for name in ("relation_bwd", "relation_bwd_prepare", "relation_bwd_main", "relation_bwd_finish"):
            getattr(lib, name).argtypes = _BWD_ARGTYPES
            getattr(lib, name).restype = ctypes.c_int
        lib.relation_bwd_noalloc.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                             _VP]
        lib.relation_bwd_noalloc.restype = ctypes.c_int
        lib.relation_step_host_device_bytes.argtypes = [ctypes.POINTER(Problem), ctypes.c_int]
        lib.relation_step_host_device_bytes.restype = ctypes.c_size_t
        lib.relation_step_host.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                           ctypes.c_int, _VP, ctypes.c_size_t, _VP]
        lib.relation_step_host.restype = ctypes.c_int
        lib.relation_bwd_workspace_bytes.argtypes = [ctypes.POINTER(Problem)]
        lib.relation_bwd_workspace_bytes.restype = ctypes.c_size_t
        lib.relation_prologue_fwd.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, ctypes.c_int,
                                              ctypes.c_float, _VP, _VP, _VP, _VP, _VP]
        lib.relation_prologue_fwd.restype = ctypes.c_int
        lib.relation_prologue_bwd.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, ctypes.c_int,
                                              ctypes.c_float, _VP, _VP, _VP, _VP, _VP, _VP]
        lib.relation_prologue_bwd.restype = ctypes.c_int
        lib.relation_fwd_prologue.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, ctypes.c_int,
                                              ctypes.c_float, _VP, _VP, _VP, _VP]
        lib.relation_fwd_prologue.restype = ctypes.c_int
        lib.relation_bwd_prologue_workspace_bytes.argtypes = [ctypes.POINTER(Problem)]
        lib.relation_bwd_prologue_workspace_bytes.restype = ctypes.c_size_t
        lib.relation_bwd_prologue.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, ctypes.c_int,
                                              ctypes.c_float, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                              ctypes.c_size_t, _VP]
        lib.relation_bwd_prologue.restype = ctypes.c_int
        lib.relation_linear_fwd_gate.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                 _VP, ctypes.c_size_t, _VP]
        lib.relation_linear_fwd_gate.restype = ctypes.c_int
        lib.relation_linear_bwd_gate.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                                 _VP, _VP, _VP, _VP, _VP, ctypes.c_int, _VP, ctypes.c_size_t, _VP]
        lib.relation_linear_bwd_gate.restype = ctypes.c_int
        lib.relation_decode_workspace_bytes.argtypes = [ctypes.POINTER(Problem)]
        lib.relation_decode_workspace_bytes.restype = ctypes.c_size_t
        lib.relation_decode.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, ctypes.c_int, _VP, _VP,
                                        _VP, ctypes.c_size_t, _VP]
        lib.relation_decode.restype = ctypes.c_int
        lib.relation_linear_workspace_bytes.argtypes = [ctypes.POINTER(Problem)]
        lib.relation_linear_workspace_bytes.restype = ctypes.c_size_t
        lib.relation_linear_fwd.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            ctypes.c_size_t, _VP]
        lib.relation_linear_fwd.restype = ctypes.c_int
        lib.relation_linear_bwd.argtypes = [ctypes.POINTER(Problem), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                            ctypes.c_int, _VP, ctypes.c_size_t, _VP]
        lib.relation_linear_bwd.restype = ctypes.c_int
        lib.relation_selftest_wait_timeout.argtypes = [ctypes.c_uint32, _VP]
        lib.relation_selftest_wait_timeout.restype = ctypes.c_int
        lib.relation_check_device_status.argtypes = []
        lib.relation_check_device_status.restype = ctypes.c_int
        lib.relation_last_launch_count.argtypes = []
        lib.relation_last_launch_count.restype = ctypes.c_int
        lib.relation_status_string.argtypes = [ctypes.c_int]
        lib.relation_status_string.restype = ctypes.c_char_p
        lib.relation_abi_version.argtypes = []
        lib.relation_abi_version.restype = ctypes.c_int
        _lib = lib
        return lib


def declared_symbols() -> list[str]:
    """Entry points declared in include/*.h."""
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include")
    names = []
    for fn in sorted(os.listdir(inc)):
        if fn.endswith(".h"):
            text = open(os.path.join(inc, fn)).read()
            names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(relation_[a-z0-9_]+)\s*\(", text, re.M)
    return sorted(set(names))


def _ptr(t) -> int | None:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("Relation tensors must be CUDA tensors")
    if not t.is_contiguous():
        raise ValueError("Relation tensors must be contiguous [B, H, T, d_h]")
    return t.data_ptr()


def _host_ptr(t) -> int | None:
    if t is None:
        return None
    if t.is_cuda:
        raise ValueError("relation_step_host takes host tensors")
    if not t.is_contiguous():
        raise ValueError("Relation tensors must be contiguous")
    return t.data_ptr()


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _check(code: int, what: str) -> None:
    if code != 0:
        msg = load().relation_status_string(code).decode()
        raise RelationError(code, what, msg)


def problem_for(t: torch.Tensor, tau_S: float, lam: float, causal: bool, layout: int = RELATION_LAYOUT_BHTD) -> Problem:
    """Problem for operand tensors shaped [B, H, T, d_h] (BHTD) or [B, T, H, d_h] (BTHD)."""
    if t.dim() != 4:
        raise ValueError("expected 4-D operand tensors")
    if t.dtype == torch.bfloat16:
        dt = RELATION_BF16
    elif t.dtype == torch.float32:
        dt = RELATION_F32
    else:
        raise ValueError(f"unsupported dtype {t.dtype}")
    if layout == RELATION_LAYOUT_BHTD:
        B, H, T, d = t.shape
    elif layout == RELATION_LAYOUT_BTHD:
        B, T, H, d = t.shape
    else:
        raise ValueError(f"unknown layout {layout}")
    return Problem(B, H, T, d, dt, float(tau_S), float(lam), 1 if causal else 0, int(layout))


# ------------------------------------------------------------------ C-ABI calls
def relation_fwd(prob: Problem, P1, P2, V, Y, L=None, stream=None) -> None:
    _check(load().relation_fwd(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(V), _ptr(Y), _ptr(L),
                               _stream_ptr(stream)), "relation_fwd")


def relation_selftest_wait_timeout(limit_ms: int, stream=None) -> None:
    _check(load().relation_selftest_wait_timeout(int(limit_ms), _stream_ptr(stream)), "relation_selftest_wait_timeout")


def relation_fwd_workspace_bytes(prob: Problem) -> int:
    return int(load().relation_fwd_workspace_bytes(ctypes.byref(prob)))


def relation_fwd_ws(prob: Problem, P1, P2, V, Y, L=None, workspace=None, stream=None) -> None:
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().relation_fwd_ws(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(V), _ptr(Y), _ptr(L), _ptr(workspace),
                                  nbytes, _stream_ptr(stream)), "relation_fwd_ws")


def relation_bwd_workspace_bytes(prob: Problem) -> int:
    return int(load().relation_bwd_workspace_bytes(ctypes.byref(prob)))


def _bwd_call(name, prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream):
    fn = getattr(load(), name)
    _check(fn(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(V), _ptr(Y), _ptr(L), _ptr(dY), _ptr(dP1), _ptr(dP2),
              _ptr(dV), _ptr(dlambda), _ptr(workspace), workspace.numel() * workspace.element_size(),
              _stream_ptr(stream)), name)


def relation_bwd(prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream=None) -> None:
    _bwd_call("relation_bwd", prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream)


def relation_bwd_prepare(prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream=None) -> None:
    _bwd_call("relation_bwd_prepare", prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream)


def relation_bwd_main(prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream=None) -> None:
    _bwd_call("relation_bwd_main", prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream)


def relation_bwd_finish(prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream=None) -> None:
    _bwd_call("relation_bwd_finish", prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, workspace, stream)


def relation_bwd_noalloc(prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlambda, stream=None) -> None:
    """relation_bwd with the library's built-in scratch array as workspace (no allocation)."""
    _check(load().relation_bwd_noalloc(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(V), _ptr(Y), _ptr(L), _ptr(dY),
                                       _ptr(dP1), _ptr(dP2), _ptr(dV), _ptr(dlambda), _stream_ptr(stream)),
           "relation_bwd_noalloc")


def relation_step_host_device_bytes(prob: Problem, chunks: int) -> int:
    return int(load().relation_step_host_device_bytes(ctypes.byref(prob), int(chunks)))


def relation_step_host(prob, P1, P2, V, dY, Y, L, dP1, dP2, dV, dlambda, chunks, device_buffer, stream=None) -> None:
    """Host tensors in and out (pinned for overlap); device_buffer a CUDA tensor of
    relation_step_host_device_bytes(prob, chunks) bytes."""
    _check(load().relation_step_host(ctypes.byref(prob), _host_ptr(P1), _host_ptr(P2), _host_ptr(V), _host_ptr(dY),
                                     _host_ptr(Y), _host_ptr(L), _host_ptr(dP1), _host_ptr(dP2), _host_ptr(dV),
                                     _host_ptr(dlambda), int(chunks), _ptr(device_buffer),
                                     device_buffer.numel() * device_buffer.element_size(), _stream_ptr(stream)),
           "relation_step_host")


def relation_decode_workspace_bytes(prob: Problem) -> int:
    return int(load().relation_decode_workspace_bytes(ctypes.byref(prob)))


def relation_decode(prob, P1_new, P2_new, V_new, P2_cache, V_cache, positions, append, Y, L, workspace,
                    stream=None) -> None:
    _check(load().relation_decode(ctypes.byref(prob), _ptr(P1_new), _ptr(P2_new), _ptr(V_new), _ptr(P2_cache),
                                  _ptr(V_cache), _ptr(positions), int(append), _ptr(Y), _ptr(L), _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "relation_decode")


def relation_prologue_fwd(prob, X1, X2, I, theta, pairing, rope_base, pos0, P1, P2, I_mixed, stream=None) -> None:
    _check(load().relation_prologue_fwd(ctypes.byref(prob), _ptr(X1), _ptr(X2), _ptr(I), _ptr(theta), int(pairing),
                                        float(rope_base), _ptr(pos0), _ptr(P1), _ptr(P2), _ptr(I_mixed),
                                        _stream_ptr(stream)), "relation_prologue_fwd")


def relation_prologue_bwd(prob, dP1, dP2, dI_mixed, I_mixed, theta, pairing, rope_base, pos0, dX1, dX2, dI, dtheta,
                          stream=None) -> None:
    _check(load().relation_prologue_bwd(ctypes.byref(prob), _ptr(dP1), _ptr(dP2), _ptr(dI_mixed), _ptr(I_mixed),
                                        _ptr(theta), int(pairing), float(rope_base), _ptr(pos0), _ptr(dX1),
                                        _ptr(dX2), _ptr(dI), _ptr(dtheta), _stream_ptr(stream)),
           "relation_prologue_bwd")


def relation_fwd_prologue(prob, X1, X2, I, theta, pairing, rope_base, pos0, Y, L=None, stream=None) -> None:
    _check(load().relation_fwd_prologue(ctypes.byref(prob), _ptr(X1), _ptr(X2), _ptr(I), _ptr(theta), int(pairing),
                                        float(rope_base), _ptr(pos0), _ptr(Y), _ptr(L), _stream_ptr(stream)),
           "relation_fwd_prologue")


def relation_bwd_prologue_workspace_bytes(prob: Problem) -> int:
    return int(load().relation_bwd_prologue_workspace_bytes(ctypes.byref(prob)))


def relation_bwd_prologue(prob, X1, X2, I, theta, pairing, rope_base, pos0, Y, L, dY, dX1, dX2, dI, dtheta, dlambda,
                          workspace, stream=None) -> None:
    nbytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(load().relation_bwd_prologue(ctypes.byref(prob), _ptr(X1), _ptr(X2), _ptr(I), _ptr(theta), int(pairing),
                                        float(rope_base), _ptr(pos0), _ptr(Y), _ptr(L), _ptr(dY), _ptr(dX1),
                                        _ptr(dX2), _ptr(dI), _ptr(dtheta), _ptr(dlambda), _ptr(workspace), nbytes,
                                        _stream_ptr(stream)), "relation_bwd_prologue")


def fused_prologue_step(X1, X2, I, theta, pairing: int, rope_base: float, tau_S: float, lam: float, dY,
                        causal: bool = True, pos0=None, layout: int = RELATION_LAYOUT_BHTD, workspace=None,
                        stream=None):
    """Forward and backward of the operator with its input prologue fused into the kernels'
    loads; allocates the outputs (and the workspace unless given) and returns
    (Y, L, dX1, dX2, dI, dtheta, dlambda)."""
    prob = problem_for(X1, tau_S, lam, causal, layout)
    Y = torch.empty_like(I)
    L = torch.empty((prob.B, prob.H, prob.T), dtype=torch.float32, device=X1.device)
    relation_fwd_prologue(prob, X1, X2, I, theta, pairing, rope_base, pos0, Y, L, stream)
    dX1, dX2, dI = torch.empty_like(X1), torch.empty_like(X2), torch.empty_like(I)
    dtheta = torch.empty(prob.H // 2, dtype=torch.float32, device=X1.device)
    dlam = torch.empty(1, dtype=torch.float32, device=X1.device)
    if workspace is None:
        n = relation_bwd_prologue_workspace_bytes(prob)
        workspace = torch.empty((n + 3) // 4, dtype=torch.float32, device=X1.device)
    relation_bwd_prologue(prob, X1, X2, I, theta, pairing, rope_base, pos0, Y, L, dY, dX1, dX2, dI, dtheta, dlam,
                          workspace, stream)
    return Y, L, dX1, dX2, dI, dtheta, dlam


def relation_linear_workspace_bytes(prob: Problem) -> int:
    return int(load().relation_linear_workspace_bytes(ctypes.byref(prob)))


def relation_linear_fwd(prob, P1, P2, I, G, Y, state, workspace, stream=None) -> None:
    _check(load().relation_linear_fwd(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(I), _ptr(G), _ptr(Y),
                                      _ptr(state), _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream_ptr(stream)), "relation_linear_fwd")


def relation_linear_bwd(prob, P1, P2, I, G, dY, dP1, dP2, dI, dG, states_from_forward, workspace,
                        stream=None) -> None:
    _check(load().relation_linear_bwd(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(I), _ptr(G), _ptr(dY), _ptr(dP1),
                                      _ptr(dP2), _ptr(dI), _ptr(dG), int(states_from_forward), _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "relation_linear_bwd")


def relation_linear_fwd_gate(prob, P1, P2, I, R, A_log, dt_bias, Y, state, workspace, stream=None) -> None:
    _check(load().relation_linear_fwd_gate(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(I), _ptr(R), _ptr(A_log),
                                           _ptr(dt_bias), _ptr(Y), _ptr(state), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "relation_linear_fwd_gate")


def relation_linear_bwd_gate(prob, P1, P2, I, R, A_log, dt_bias, dY, dP1, dP2, dI, dR, dA_log, d_dt_bias,
                             states_from_forward, workspace, stream=None) -> None:
    _check(load().relation_linear_bwd_gate(ctypes.byref(prob), _ptr(P1), _ptr(P2), _ptr(I), _ptr(R), _ptr(A_log),
                                           _ptr(dt_bias), _ptr(dY), _ptr(dP1), _ptr(dP2), _ptr(dI), _ptr(dR),
                                           _ptr(dA_log), _ptr(d_dt_bias), int(states_from_forward), _ptr(workspace),
                                           workspace.numel() * workspace.element_size(), _stream_ptr(stream)),
           "relation_linear_bwd_gate")


def linear_gate_fwd_bwd(P1, P2, I, R, A_log, dt_bias, dY, tau_S: float, layout: int = RELATION_LAYOUT_BHTD,
                        stream=None):
    """Gated Linear Relation forward and backward (states reused); returns
    (Y, dP1, dP2, dI, dR, dA_log, d_dt_bias)."""
    prob = problem_for(P1, tau_S, 0.0, True, layout)
    ws = linear_workspace(prob, P1.device)
    Y = torch.empty_like(I)
    relation_linear_fwd_gate(prob, P1, P2, I, R, A_log, dt_bias, Y, None, ws, stream)
    dP1, dP2, dI, dR = torch.empty_like(P1), torch.empty_like(P2), torch.empty_like(I), torch.empty_like(R)
    dA, dB = torch.empty_like(A_log), torch.empty_like(dt_bias)
    relation_linear_bwd_gate(prob, P1, P2, I, R, A_log, dt_bias, dY, dP1, dP2, dI, dR, dA, dB, True, ws, stream)
    return Y, dP1, dP2, dI, dR, dA, dB


def relation_check_device_status() -> int:
    return int(load().relation_check_device_status())


def relation_last_launch_count() -> int:
    return int(load().relation_last_launch_count())


def relation_status_string(code: int) -> str:
    return load().relation_status_string(code).decode()


def relation_abi_version() -> int:
    return int(load().relation_abi_version())


# ------------------------------------------------------- tensor-level helpers
def fwd_workspace(prob: Problem, device):
    """Workspace tensor for relation_fwd_ws, or None when the problem needs none."""
    n = relation_fwd_workspace_bytes(prob)
    return torch.empty((n + 3) // 4, dtype=torch.float32, device=device) if n else None


def fwd(P1, P2, V, tau_S: float, lam: float, causal: bool = True, stream=None, want_L: bool = True,
        layout: int = RELATION_LAYOUT_BHTD, workspace=None, use_workspace: bool = True):
    """Allocates Y (and L [B, H, T]) and runs the forward; returns (Y, L).  Head widths that
    need a workspace (bf16 d_h = 60) get one (allocated here unless given) and run through
    relation_fwd_ws; use_workspace=False runs relation_fwd instead."""
    prob = problem_for(P1, tau_S, lam, causal, layout)
    Y = torch.empty_like(V)
    L = torch.empty((prob.B, prob.H, prob.T), dtype=torch.float32, device=P1.device) if want_L else None
    if use_workspace and relation_fwd_workspace_bytes(prob):
        if workspace is None:
            workspace = fwd_workspace(prob, P1.device)
        relation_fwd_ws(prob, P1, P2, V, Y, L, workspace, stream)
    else:
        relation_fwd(prob, P1, P2, V, Y, L, stream)
    return Y, L


def linear_workspace(prob: Problem, device) -> torch.Tensor:
    """Workspace tensor for relation_linear_fwd / relation_linear_bwd."""
    n = relation_linear_workspace_bytes(prob)
    return torch.empty(max(1, (n + 3) // 4), dtype=torch.float32, device=device)


def linear_fwd(P1, P2, I, G, tau_S: float, layout: int = RELATION_LAYOUT_BHTD, want_state: bool = False,
               stream=None, workspace=None):
    """Linear Relation forward; allocates Y (and the final state [B, H, d, d]); returns (Y, state)."""
    prob = problem_for(P1, tau_S, 0.0, True, layout)
    Y = torch.empty_like(I)
    state = (torch.empty((prob.B, prob.H, prob.d_h, prob.d_h), dtype=torch.float32, device=P1.device)
             if want_state else None)
    if workspace is None:
        workspace = linear_workspace(prob, P1.device)
    relation_linear_fwd(prob, P1, P2, I, G, Y, state, workspace, stream)
    return Y, state


def linear_bwd(P1, P2, I, G, dY, tau_S: float, layout: int = RELATION_LAYOUT_BHTD, stream=None, workspace=None,
               states_from_forward: bool = False):
    """Linear Relation backward; allocates and returns (dP1, dP2, dI, dG).  states_from_forward:
    ``workspace`` still holds what linear_fwd left in it for the same inputs."""
    prob = problem_for(P1, tau_S, 0.0, True, layout)
    dP1, dP2, dI, dG = torch.empty_like(P1), torch.empty_like(P2), torch.empty_like(I), torch.empty_like(G)
    if workspace is None:
        if states_from_forward:
            raise ValueError("states_from_forward needs the forward's workspace")
        workspace = linear_workspace(prob, P1.device)
    relation_linear_bwd(prob, P1, P2, I, G, dY, dP1, dP2, dI, dG, states_from_forward, workspace, stream)
    return dP1, dP2, dI, dG


def decode(P1_new, P2_new, V_new, P2_cache, V_cache, positions, tau_S: float, lam: float, append: bool = True,
           layout: int = RELATION_LAYOUT_BHTD, stream=None, workspace=None):
    """One Relation Cache step; allocates Y [B, H, d_h] and L [B, H]; returns (Y, L)."""
    B, H, d = P1_new.shape
    T = P2_cache.shape[2] if layout == RELATION_LAYOUT_BHTD else P2_cache.shape[1]
    dt = RELATION_BF16 if P1_new.dtype == torch.bfloat16 else RELATION_F32
    prob = Problem(B, H, T, d, dt, float(tau_S), float(lam), 1, int(layout))
    Y = torch.empty_like(P1_new)
    L = torch.empty((B, H), dtype=torch.float32, device=P1_new.device)
    if workspace is None:
        workspace = torch.empty((relation_decode_workspace_bytes(prob) + 3) // 4, dtype=torch.float32,
                                device=P1_new.device)
    relation_decode(prob, P1_new, P2_new, V_new, P2_cache, V_cache, positions, append, Y, L, workspace, stream)
    return Y, L


def step_host(P1, P2, V, dY, tau_S: float, lam: float, causal: bool = True, chunks: int = 1, out=None,
              device_buffer=None, want_L: bool = False, stream=None, layout: int = RELATION_LAYOUT_BHTD):
    """relation_step_host on host tensors; allocates what is not given (pinned host outputs,
    the device buffer).  Returns (Y, L or None, dP1, dP2, dV, dlambda) as host tensors."""
    prob = problem_for(P1, tau_S, lam, causal, layout)
    if out is None:
        out = tuple(torch.empty(P1.shape, dtype=P1.dtype).pin_memory() for _ in range(4))
    Y, dP1, dP2, dV = out
    L = torch.empty((prob.B, prob.H, prob.T), dtype=torch.float32).pin_memory() if want_L else None
    dlam = torch.empty(1, dtype=torch.float32).pin_memory()
    if device_buffer is None:
        nbytes = relation_step_host_device_bytes(prob, chunks)
        device_buffer = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device="cuda")
    relation_step_host(prob, P1, P2, V, dY, Y, L, dP1, dP2, dV, dlam, chunks, device_buffer, stream)
    return Y, L, dP1, dP2, dV, dlam


def bwd(P1, P2, V, Y, L, dY, tau_S: float, lam: float, causal: bool = True, stream=None, workspace=None,
        layout: int = RELATION_LAYOUT_BHTD):
    """Allocates the gradients and workspace and runs relation_bwd; returns (dP1, dP2, dV, dlambda)."""
    prob = problem_for(P1, tau_S, lam, causal, layout)
    dP1, dP2, dV = torch.empty_like(P1), torch.empty_like(P2), torch.empty_like(V)
    dlam = torch.empty(1, dtype=torch.float32, device=P1.device)
    if workspace is None:
        nbytes = relation_bwd_workspace_bytes(prob)
        workspace = torch.empty((nbytes + 3) // 4, dtype=torch.float32, device=P1.device)
    relation_bwd(prob, P1, P2, V, Y, L, dY, dP1, dP2, dV, dlam, workspace, stream)
    return dP1, dP2, dV, dlam
