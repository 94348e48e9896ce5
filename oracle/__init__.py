"""Float64 CPU oracle for the Full Relation operator.

TEST INFRASTRUCTURE ONLY.  The tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product library never does.  The
arithmetic lives in ``relation_oracle.c`` (plain C, float64, OpenMP over
independent heads or rows); this module only compiles it with gcc and
marshals arrays.

Definition followed: "Ask Self, Ask Others: Relation Is All You Need",
Sec. 3.1 eq.(1)-(3) and Appendix A.1; the second (FlashRelation) path follows
Sec. 5.1 eq.(12)-(14) and Appendix A.3.  See the C file's header for the
formulas and for the backward derived by the chain rule.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "relation_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "librelation_oracle.so")
_lock = threading.Lock()
_lib = None


class _Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int64),
        ("H", ctypes.c_int64),
        ("T", ctypes.c_int64),
        ("d", ctypes.c_int64),
        ("tau_S", ctypes.c_double),
        ("lam", ctypes.c_double),
        ("causal", ctypes.c_int),
    ]


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/librelation_oracle.so``."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    fresh = os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER(_Problem)
            dp = ctypes.POINTER(ctypes.c_double)
            ip = ctypes.POINTER(ctypes.c_int64)
            i64 = ctypes.c_int64
            lib.relation_oracle_fwd.argtypes = [P, dp, dp, dp, dp, dp]
            lib.relation_oracle_fwd_rows.argtypes = [P, dp, dp, dp, i64, ip, ip, dp, dp]
            lib.relation_oracle_bwd.argtypes = [P, dp, dp, dp, dp, dp, dp, dp, dp]
            lib.relation_oracle_row_stats.argtypes = [P, dp, dp, dp, dp, i64, dp, dp]
            lib.relation_oracle_bwd_cols.argtypes = [P, dp, dp, dp, dp, i64, dp, dp, i64, ip, dp, dp]
            lib.relation_oracle_bwd_rows.argtypes = [P, dp, dp, dp, dp, i64, i64, ip, dp]
            lib.relation_oracle_flash_fwd.argtypes = [P, dp, dp, dp, i64, ip, dp, dp]
            lib.relation_oracle_threads.argtypes = []
            for name in ("relation_oracle_fwd", "relation_oracle_fwd_rows", "relation_oracle_bwd",
                         "relation_oracle_row_stats", "relation_oracle_bwd_cols",
                         "relation_oracle_bwd_rows", "relation_oracle_flash_fwd",
                         "relation_oracle_threads"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def threads() -> int:
    """OpenMP threads the oracle runs with."""
    return int(_load().relation_oracle_threads())


def _f64(x) -> np.ndarray:
    """Exact upcast to a contiguous float64 array (accepts numpy or torch)."""
    if hasattr(x, "detach"):
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _dp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _ip(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def _problem(shape, tau_S, lam, causal) -> _Problem:
    if len(shape) != 4:
        raise ValueError("expected [B, H, T, d] tensors")
    B, H, T, d = shape
    return _Problem(B, H, T, d, float(tau_S), float(lam), 1 if causal else 0)


def _check(rc: int, what: str) -> None:
    if rc != 0:
        raise ValueError(f"oracle {what} failed with code {rc}")


def fwd(P1, P2, V, tau_S: float, lam: float, causal: bool = True):
    """Full forward.  Returns (Y [B,H,T,d], L [B,H,T]) as float64."""
    P1, P2, V = _f64(P1), _f64(P2), _f64(V)
    if not (P1.shape == P2.shape == V.shape):
        raise ValueError("P1, P2, V shapes differ")
    prob = _problem(P1.shape, tau_S, lam, causal)
    Y = np.empty_like(V)
    L = np.empty(P1.shape[:3], dtype=np.float64)
    _check(_load().relation_oracle_fwd(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), _dp(Y), _dp(L)), "fwd")
    return Y, L


def fwd_rows(P1, P2, V, tau_S, lam, causal, heads, rows):
    """Forward of selected rows; ``heads`` index the flattened B*H axis."""
    P1, P2, V = _f64(P1), _f64(P2), _f64(V)
    prob = _problem(P1.shape, tau_S, lam, causal)
    heads = np.ascontiguousarray(heads, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = heads.size
    Y = np.empty((n, P1.shape[3]), dtype=np.float64)
    L = np.empty((n,), dtype=np.float64)
    _check(_load().relation_oracle_fwd_rows(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), n, _ip(heads),
                                            _ip(rows), _dp(Y), _dp(L)), "fwd_rows")
    return Y, L


def bwd(P1, P2, V, dY, tau_S: float, lam: float, causal: bool = True):
    """Full backward.  Returns (dP1, dP2, dV, dlambda) as float64."""
    P1, P2, V, dY = _f64(P1), _f64(P2), _f64(V), _f64(dY)
    prob = _problem(P1.shape, tau_S, lam, causal)
    dP1, dP2, dV = np.empty_like(P1), np.empty_like(P2), np.empty_like(V)
    dlam = ctypes.c_double(0.0)
    _check(_load().relation_oracle_bwd(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), _dp(dY), _dp(dP1),
                                       _dp(dP2), _dp(dV), ctypes.byref(dlam)), "bwd")
    return dP1, dP2, dV, dlam.value


def row_stats(P1, P2, V, dY, tau_S, lam, causal, head: int):
    """(L, D) of every row of one head (flattened B*H index)."""
    P1, P2, V, dY = _f64(P1), _f64(P2), _f64(V), _f64(dY)
    prob = _problem(P1.shape, tau_S, lam, causal)
    T = P1.shape[2]
    L = np.empty((T,), dtype=np.float64)
    D = np.empty((T,), dtype=np.float64)
    _check(_load().relation_oracle_row_stats(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), _dp(dY), int(head),
                                             _dp(L), _dp(D)), "row_stats")
    return L, D


def bwd_cols(P1, P2, V, dY, tau_S, lam, causal, head: int, L, D, cols):
    """(dP2, dV) rows for selected columns j of one head, from that head's L and D."""
    P1, P2, V, dY = _f64(P1), _f64(P2), _f64(V), _f64(dY)
    L, D = _f64(L), _f64(D)
    prob = _problem(P1.shape, tau_S, lam, causal)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    n = cols.size
    dP2 = np.empty((n, P1.shape[3]), dtype=np.float64)
    dV = np.empty((n, P1.shape[3]), dtype=np.float64)
    _check(_load().relation_oracle_bwd_cols(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), _dp(dY), int(head),
                                            _dp(L), _dp(D), n, _ip(cols), _dp(dP2), _dp(dV)), "bwd_cols")
    return dP2, dV


def bwd_rows(P1, P2, V, dY, tau_S, lam, causal, head: int, rows):
    """dP1 rows for selected rows i of one head."""
    P1, P2, V, dY = _f64(P1), _f64(P2), _f64(V), _f64(dY)
    prob = _problem(P1.shape, tau_S, lam, causal)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    n = rows.size
    dP1 = np.empty((n, P1.shape[3]), dtype=np.float64)
    _check(_load().relation_oracle_bwd_rows(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), _dp(dY), int(head), n,
                                            _ip(rows), _dp(dP1)), "bwd_rows")
    return dP1


def flash_fwd(P1, P2, V, tau_S: float, lam: float, tile_sizes):
    """Second path (FlashRelation tiled Exchange scan), causal only; cross-check use."""
    P1, P2, V = _f64(P1), _f64(P2), _f64(V)
    prob = _problem(P1.shape, tau_S, lam, True)
    tiles = np.ascontiguousarray(tile_sizes, dtype=np.int64)
    Y = np.empty_like(V)
    L = np.empty(P1.shape[:3], dtype=np.float64)
    _check(_load().relation_oracle_flash_fwd(ctypes.byref(prob), _dp(P1), _dp(P2), _dp(V), tiles.size,
                                             _ip(tiles), _dp(Y), _dp(L)), "flash_fwd")
    return Y, L
