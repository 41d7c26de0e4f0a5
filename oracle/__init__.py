"""fp64 CPU oracle for Fibottention's per-head sparse self-attention.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It compiles and
loads ``fibatt_oracle.c`` (plain C, fp64) and shares no code with the CUDA
library in ``sparse_head_self_gb300``; neither side imports the other.

Sources: "Fibottention: Inceptive Visual Representation Learning with Diverse
Attention Across Heads" (arXiv 2406.19391) Sec. 3 (support set, Wythoff rows,
window schedule) and the Fibottention project README, Algorithms 1-3.

Every function here is pinned by ``tests/test_oracle_pins.py`` to something
other than itself (closed forms, an independent Zeckendorf construction of the
Wythoff array, dense library attention, finite differences).
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fibatt_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_i32p = ctypes.POINTER(ctypes.c_int32)
_f64p = ctypes.POINTER(ctypes.c_double)
_u8p = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, -O2).

    OpenMP is used when the compiler supports it; otherwise the oracle runs
    serially.  Returns the library path.
    """
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("oracle build needs a C compiler (gcc)")
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    base = [cc, "-O2", "-fPIC", "-shared", "-std=c11", "-o", tmp, _SRC, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True,
                       capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        lib.orc_set_threads.argtypes = [ctypes.c_int]
        lib.orc_set_threads.restype = ctypes.c_int
        lib.orc_max_threads.restype = ctypes.c_int
        lib.orc_isqrt.argtypes = [ctypes.c_int64]
        lib.orc_isqrt.restype = ctypes.c_int64
        lib.orc_floor_mul_phi.argtypes = [ctypes.c_int64]
        lib.orc_floor_mul_phi.restype = ctypes.c_int64
        lib.orc_wythoff_row.argtypes = [ctypes.c_int64, _i64p, _i64p]
        lib.orc_wythoff_row.restype = ctypes.c_int
        lib.orc_fib_list.argtypes = [ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _i64p,
                                     ctypes.c_int]
        lib.orc_fib_list.restype = ctypes.c_int
        lib.orc_window.argtypes = [ctypes.c_int64] * 4
        lib.orc_window.restype = ctypes.c_int64
        lib.orc_in_support.argtypes = [ctypes.c_int64, ctypes.c_int64, _i64p, ctypes.c_int,
                                       ctypes.c_int64, ctypes.c_int]
        lib.orc_in_support.restype = ctypes.c_int
        lib.orc_support_mask.argtypes = [ctypes.c_int64, _i64p, ctypes.c_int, ctypes.c_int64,
                                         ctypes.c_int, _u8p]
        lib.orc_support_mask.restype = ctypes.c_int64
        lib.orc_signed_table.argtypes = [ctypes.c_int64, _i64p, ctypes.c_int, ctypes.c_int64,
                                         ctypes.c_int, _i32p, ctypes.c_int]
        lib.orc_signed_table.restype = ctypes.c_int
        lib.orc_fwd_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, _f64p,
                                     _i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_double, _i64p, ctypes.c_int64, _f64p, _f64p]
        lib.orc_fwd_rows.restype = None
        lib.orc_bwd_rows.argtypes = [ctypes.c_int64, ctypes.c_int64, _f64p, _f64p, _f64p, _f64p,
                                     _i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_double, _i64p, ctypes.c_int64, _i64p,
                                     ctypes.c_int64, _f64p, _f64p, _f64p]
        lib.orc_bwd_rows.restype = None
        _lib = lib
        return lib


def _ptr(a: np.ndarray | None, typ):
    if a is None:
        return ctypes.cast(None, typ)
    return a.ctypes.data_as(typ)


def set_threads(n: int) -> int:
    """Host threads used by the oracle's row loops; returns the count in effect."""
    return _load().orc_set_threads(int(n))


def max_threads() -> int:
    return _load().orc_max_threads()


# ------------------------------------------------------------------ integers

def isqrt(n: int) -> int:
    return _load().orc_isqrt(int(n))


def floor_mul_phi(n: int) -> int:
    return _load().orc_floor_mul_phi(int(n))


def wythoff_row(i: int) -> tuple[int, int]:
    """(a_i, b_i): the first two entries of row i (1-based) of the Wythoff array."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    if _load().orc_wythoff_row(int(i), ctypes.byref(a), ctypes.byref(b)) != 0:
        raise ValueError(f"Wythoff row index out of range: {i}")
    return a.value, b.value


def fib_list(a: int, b: int, w: int) -> list[int]:
    """Algorithm 1 of the project README: [a, b, ...] extended while last < w."""
    lib = _load()
    n = lib.orc_fib_list(int(a), int(b), int(w), _ptr(None, _i64p), 0)
    if n < 0:
        raise ValueError(f"Fib({a},{b}) does not terminate or is invalid")
    out = np.zeros(n, dtype=np.int64)
    lib.orc_fib_list(int(a), int(b), int(w), _ptr(out, _i64p), n)
    return [int(x) for x in out]


def window(i: int, h: int, w_min: int, w_max: int) -> int:
    """Window of head i (1-based) among h heads (Fibottention Sec. 3.2)."""
    return _load().orc_window(int(i), int(h), int(w_min), int(w_max))


def windows(h: int, w_min: int, w_max: int) -> list[int]:
    return [window(i, h, w_min, w_max) for i in range(1, h + 1)]


# ------------------------------------------------------------------- support

class Head:
    """One head's support: distance set S, window w, diagonal flag, and the
    optional global first token (README Algorithm 2: row 0 and column 0 of
    the mask are all ones)."""

    def __init__(self, S, w: int, diag: bool, global_token: bool = False):
        self.S = np.ascontiguousarray(np.asarray(list(S), dtype=np.int64))
        self.w = int(w)
        self.diag = 1 if diag else 0
        self.global_token = bool(global_token)

    @classmethod
    def fibottention(cls, a: int, b: int, w: int, diag: bool, global_token: bool = False) -> "Head":
        return cls(fib_list(a, b, w), w, diag, global_token)

    def _args(self):
        return _ptr(self.S, _i64p), int(self.S.size), self.w, self.diag | (2 if self.global_token else 0)


def wythoff_heads(H: int, N: int, w_min: int, w_max: int, diag: bool,
                  first_row: int = 1, global_token: bool = False) -> list[Head]:
    """Heads 1..H on Wythoff rows first_row.. with the linear window schedule."""
    heads = []
    for i in range(1, H + 1):
        a, b = wythoff_row(first_row + i - 1)
        heads.append(Head.fibottention(a, b, window(i, H, w_min, w_max), diag, global_token))
    return heads


def in_support(j: int, k: int, head: Head) -> bool:
    S, nS, w, diag = head._args()
    return bool(_load().orc_in_support(int(j), int(k), S, nS, w, diag))


def support_mask(N: int, head: Head) -> np.ndarray:
    mask = np.zeros((N, N), dtype=np.uint8)
    S, nS, w, diag = head._args()
    _load().orc_support_mask(int(N), S, nS, w, diag, _ptr(mask, _u8p))
    return mask


def support_size(N: int, head: Head) -> int:
    S, nS, w, diag = head._args()
    return int(_load().orc_support_mask(int(N), S, nS, w, diag, _ptr(None, _u8p)))


def signed_table(N: int, head: Head) -> np.ndarray:
    lib = _load()
    S, nS, w, diag = head._args()
    n = lib.orc_signed_table(int(N), S, nS, w, diag, _ptr(None, _i32p), 0)
    out = np.zeros(n, dtype=np.int32)
    lib.orc_signed_table(int(N), S, nS, w, diag, _ptr(out, _i32p), n)
    return out


# --------------------------------------------------------------- attention

def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().to("cpu").double().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _rows(rows):
    if rows is None:
        return None
    return np.ascontiguousarray(np.asarray(rows, dtype=np.int64))


def fwd_head(Q, K, V, head: Head, scale: float, rows=None):
    """Forward of one head: Q, K, V are [N, Dh]; returns (O [n, Dh], LSE [n])."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    N, Dh = Q.shape
    r = _rows(rows)
    n = N if r is None else r.size
    O = np.zeros((n, Dh), dtype=np.float64)
    L = np.zeros(n, dtype=np.float64)
    S, nS, w, diag = head._args()
    _load().orc_fwd_rows(N, Dh, _ptr(Q, _f64p), _ptr(K, _f64p), _ptr(V, _f64p), S, nS, w, diag,
                         float(scale), _ptr(r, _i64p), n, _ptr(O, _f64p), _ptr(L, _f64p))
    return O, L


def bwd_head(Q, K, V, dO, head: Head, scale: float, qrows=None, krows=None,
             want_dq: bool = True, want_dkv: bool = True):
    """Backward of one head for L = sum(dO * O): returns (dQ, dK, dV) on the listed rows."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    N, Dh = Q.shape
    qr, kr = _rows(qrows), _rows(krows)
    nq = N if qr is None else qr.size
    nk = N if kr is None else kr.size
    dQ = np.zeros((nq, Dh)) if want_dq else None
    dK = np.zeros((nk, Dh)) if want_dkv else None
    dV = np.zeros((nk, Dh)) if want_dkv else None
    S, nS, w, diag = head._args()
    _load().orc_bwd_rows(N, Dh, _ptr(Q, _f64p), _ptr(K, _f64p), _ptr(V, _f64p), _ptr(dO, _f64p),
                         S, nS, w, diag, float(scale), _ptr(qr, _i64p), nq, _ptr(kr, _i64p), nk,
                         _ptr(dQ, _f64p), _ptr(dK, _f64p), _ptr(dV, _f64p))
    return dQ, dK, dV


def fwd(Q, K, V, heads: list[Head], scale: float, rows=None):
    """Forward over [B, H, N, Dh] tensors; head h of every batch uses heads[h].

    Returns (O [B, H, n, Dh], LSE [B, H, n]) in fp64 on the listed query rows.
    """
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, Dh = Q.shape
    assert len(heads) == H
    n = N if rows is None else len(rows)
    O = np.zeros((B, H, n, Dh))
    L = np.zeros((B, H, n))
    for b in range(B):
        for h in range(H):
            O[b, h], L[b, h] = fwd_head(Q[b, h], K[b, h], V[b, h], heads[h], scale, rows)
    return O, L


def bwd(Q, K, V, dO, heads: list[Head], scale: float, qrows=None, krows=None):
    """Backward over [B, H, N, Dh] tensors; returns (dQ, dK, dV) in fp64."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, Dh = Q.shape
    nq = N if qrows is None else len(qrows)
    nk = N if krows is None else len(krows)
    dQ = np.zeros((B, H, nq, Dh))
    dK = np.zeros((B, H, nk, Dh))
    dV = np.zeros((B, H, nk, Dh))
    for b in range(B):
        for h in range(H):
            dQ[b, h], dK[b, h], dV[b, h] = bwd_head(Q[b, h], K[b, h], V[b, h], dO[b, h],
                                                   heads[h], scale, qrows, krows)
    return dQ, dK, dV
