"""Python binding of libfibatt: same names as the C ABI, argument marshalling only.

Every step of the attention runs in the library's CUDA kernels; torch is used
for device memory, dtypes and the current stream.  There is no CPU fallback:
calls on CPU tensors are rejected.
"""
from __future__ import annotations

import ctypes

import torch

from . import _native
from ._native import FibattError, check, lib

HEAD_DIM = 64

_DTYPES = {torch.float32: _native.F32, torch.bfloat16: _native.BF16}


# ------------------------------------------------------------------ helpers

def wythoff_row(i: int) -> tuple[int, int]:
    """(a_i, b_i) of Wythoff row i (Fibottention Sec. 3.2)."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    check(lib().fibatt_wythoff_row(int(i), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def wythoff_row_modified(i: int) -> tuple[int, int]:
    """The two terms preceding Wythoff row i (README Algorithm 2, modified variant)."""
    a, b = ctypes.c_int64(), ctypes.c_int64()
    check(lib().fibatt_wythoff_row_modified(int(i), ctypes.byref(a), ctypes.byref(b)))
    return a.value, b.value


def window_schedule(h: int, w_min: int, w_max: int) -> list[int]:
    """Per-head windows w_1..w_h (Fibottention Sec. 3.2)."""
    w = (ctypes.c_int64 * h)()
    check(lib().fibatt_window_schedule(int(h), int(w_min), int(w_max), w))
    return list(w)


def _i64(xs):
    xs = [int(x) for x in xs]
    return (ctypes.c_int64 * max(1, len(xs)))(*xs)


def _i32(xs):
    xs = [int(x) for x in xs]
    return (ctypes.c_int32 * max(1, len(xs)))(*xs)


class Support:
    """Owner of a ``fibatt_support_t`` handle (host memory only)."""

    def __init__(self, handle: ctypes.c_void_p):
        self._h = handle
        H, N, total = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        check(lib().fibatt_support_info(self._h, ctypes.byref(H), ctypes.byref(N), ctypes.byref(total)))
        self.H, self.N, self.total_entries = H.value, N.value, total.value

    # -- constructors --------------------------------------------------------
    @classmethod
    def build(cls, N: int, a, b, w, include_diag: bool) -> "Support":
        """fibatt_support_build: head h uses Fib(a[h], b[h]) within window w[h]."""
        H = len(a)
        assert len(b) == H and len(w) == H
        h = ctypes.c_void_p()
        check(lib().fibatt_support_build(H, int(N), _i64(a), _i64(b), _i64(w), int(bool(include_diag)),
                                         ctypes.byref(h)))
        return cls(h)

    @classmethod
    def from_distances(cls, N: int, distances: list, include_diag: bool) -> "Support":
        """fibatt_support_build_distances: head h attends |j-k| in distances[h]."""
        counts = [len(d) for d in distances]
        flat = [int(x) for d in distances for x in d]
        h = ctypes.c_void_p()
        check(lib().fibatt_support_build_distances(len(distances), int(N), _i32(counts), _i32(flat),
                                                   int(bool(include_diag)), ctypes.byref(h)))
        return cls(h)

    @classmethod
    def wythoff(cls, H: int, N: int, w_min: int, w_max: int, include_diag: bool,
                modified: bool = False, permutation=None) -> "Support":
        """Fibottention's layer support: head i on Wythoff row pi(i) (rows 1..H),
        windows from the linear schedule."""
        row = wythoff_row_modified if modified else wythoff_row
        ab = [row(i) for i in range(1, H + 1)]
        w = window_schedule(H, w_min, w_max)
        perm = list(range(H)) if permutation is None else [int(p) for p in permutation]
        assert sorted(perm) == list(range(H))
        return cls.build(N, [ab[p][0] for p in perm], [ab[p][1] for p in perm], [w[p] for p in perm],
                         include_diag)

    def set_global_token(self, enabled: bool = True) -> "Support":
        """fibatt_support_set_global_token: token 0 attends every key and is
        attended by every query (README Algorithm 2's class token)."""
        check(lib().fibatt_support_set_global_token(self._h, int(bool(enabled))))
        return self

    # -- queries -------------------------------------------------------------
    def tables(self):
        """(counts[H], signed offsets (CSR), pairs[H])."""
        counts = (ctypes.c_int32 * self.H)()
        offs = (ctypes.c_int32 * max(1, self.total_entries))()
        pairs = (ctypes.c_int64 * self.H)()
        check(lib().fibatt_support_get(self._h, counts, offs, pairs))
        return list(counts), list(offs)[: self.total_entries], list(pairs)

    def head_offsets(self) -> list[list[int]]:
        counts, offs, _ = self.tables()
        out, p = [], 0
        for c in counts:
            out.append(offs[p:p + c])
            p += c
        return out

    @property
    def pairs(self) -> list[int]:
        return self.tables()[2]

    def total_pairs(self, B: int = 1) -> int:
        return B * sum(self.pairs)

    def bwd_workspace_bytes(self, B: int) -> int:
        return int(lib().fibatt_bwd_workspace_bytes(self._h, int(B)))

    @property
    def handle(self) -> ctypes.c_void_p:
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().fibatt_support_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


# --------------------------------------------------------------- attention

def _check_io(name: str, t: torch.Tensor, shape, dtype, device) -> None:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (libfibatt has no CPU path)")
    if t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _stream_ptr(stream, device) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def fwd(support: Support, Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, scale: float,
        O: torch.Tensor | None = None, LSE: torch.Tensor | None = None, stream=None):
    """fibatt_fwd on [B, H, N, 64] CUDA tensors; returns (O, LSE)."""
    if Q.dim() != 4:
        raise ValueError("Q must be [B, H, N, D]")
    B, H, N, D = Q.shape
    if (H, N) != (support.H, support.N):
        raise ValueError(f"tensors have H={H}, N={N}; support has H={support.H}, N={support.N}")
    if Q.dtype not in _DTYPES:
        raise ValueError(f"dtype {Q.dtype} unsupported (float32 or bfloat16)")
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V)):
        _check_io(n, t, Q.shape, Q.dtype, dev)
    if O is None:
        O = torch.empty_like(Q)
    if LSE is None:
        LSE = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    _check_io("O", O, Q.shape, Q.dtype, dev)
    _check_io("LSE", LSE, (B, H, N), torch.float32, dev)
    check(lib().fibatt_fwd(support.handle, B, D, _DTYPES[Q.dtype], Q.data_ptr(), K.data_ptr(),
                           V.data_ptr(), float(scale), O.data_ptr(), LSE.data_ptr(),
                           _stream_ptr(stream, dev)))
    return O, LSE


def bwd(support: Support, Q, K, V, O, LSE, dO, scale: float, dQ=None, dK=None, dV=None,
        workspace: torch.Tensor | None = None, stream=None):
    """fibatt_bwd on [B, H, N, 64] CUDA tensors; returns (dQ, dK, dV)."""
    B, H, N, D = Q.shape
    if (H, N) != (support.H, support.N):
        raise ValueError(f"tensors have H={H}, N={N}; support has H={support.H}, N={support.N}")
    if Q.dtype not in _DTYPES:
        raise ValueError(f"dtype {Q.dtype} unsupported (float32 or bfloat16)")
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V), ("O", O), ("dO", dO)):
        _check_io(n, t, Q.shape, Q.dtype, dev)
    _check_io("LSE", LSE, (B, H, N), torch.float32, dev)
    dQ = torch.empty_like(Q) if dQ is None else dQ
    dK = torch.empty_like(Q) if dK is None else dK
    dV = torch.empty_like(Q) if dV is None else dV
    for n, t in (("dQ", dQ), ("dK", dK), ("dV", dV)):
        _check_io(n, t, Q.shape, Q.dtype, dev)
    need = support.bwd_workspace_bytes(B)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    check(lib().fibatt_bwd(support.handle, B, D, _DTYPES[Q.dtype], Q.data_ptr(), K.data_ptr(),
                           V.data_ptr(), O.data_ptr(), LSE.data_ptr(), dO.data_ptr(), float(scale),
                           dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), ws_ptr, ws_bytes,
                           _stream_ptr(stream, dev)))
    return dQ, dK, dV


def bwd_noalloc(support: Support, Q, K, V, O, LSE, dO, scale: float, dQ, dK, dV, stream=None):
    """fibatt_bwd_noalloc: the backward pass without any workspace argument, for
    callers that must not allocate device memory (its scratch is a fixed array
    inside the library; at most B*H*N = FIBATT_NOALLOC_MAX_ROWS rows).  The
    output tensors dQ, dK, dV are required and written in place."""
    B, H, N, D = Q.shape
    if (H, N) != (support.H, support.N):
        raise ValueError(f"tensors have H={H}, N={N}; support has H={support.H}, N={support.N}")
    if Q.dtype not in _DTYPES:
        raise ValueError(f"dtype {Q.dtype} unsupported (float32 or bfloat16)")
    dev = Q.device
    for n, t in (("Q", Q), ("K", K), ("V", V), ("O", O), ("dO", dO), ("dQ", dQ), ("dK", dK), ("dV", dV)):
        _check_io(n, t, Q.shape, Q.dtype, dev)
    _check_io("LSE", LSE, (B, H, N), torch.float32, dev)
    check(lib().fibatt_bwd_noalloc(support.handle, B, D, _DTYPES[Q.dtype], Q.data_ptr(), K.data_ptr(),
                                   V.data_ptr(), O.data_ptr(), LSE.data_ptr(), dO.data_ptr(), float(scale),
                                   dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), _stream_ptr(stream, dev)))
    return dQ, dK, dV


class FibottentionFunction(torch.autograd.Function):
    """Autograd wrapper: forward = fibatt_fwd, backward = fibatt_bwd."""

    @staticmethod
    def forward(ctx, Q, K, V, support: Support, scale: float):
        Q, K, V = Q.contiguous(), K.contiguous(), V.contiguous()
        O, LSE = fwd(support, Q, K, V, scale)
        ctx.save_for_backward(Q, K, V, O, LSE)
        ctx.support = support
        ctx.scale = scale
        return O

    @staticmethod
    def backward(ctx, dO):
        Q, K, V, O, LSE = ctx.saved_tensors
        dQ, dK, dV = bwd(ctx.support, Q, K, V, O, LSE, dO.contiguous(), ctx.scale)
        return dQ, dK, dV, None, None


def fibottention(Q, K, V, support: Support, scale: float | None = None):
    """Differentiable Fibottention attention on [B, H, N, 64] CUDA tensors."""
    if scale is None:
        scale = Q.shape[-1] ** -0.5
    return FibottentionFunction.apply(Q, K, V, support, float(scale))


__all__ = ["FibattError", "Support", "fwd", "bwd", "bwd_noalloc", "fibottention", "FibottentionFunction",
           "wythoff_row", "wythoff_row_modified", "window_schedule", "HEAD_DIM"]
