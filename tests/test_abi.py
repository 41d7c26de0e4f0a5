"""Host-side tests of libfibatt's C ABI (no GPU needed).

Covers: the library builds and exports every function include/fibatt.h
declares; support tables are bit-exact against the oracle's brute-force
support (Fibottention Sec. 3 support set); helper rows/windows match the
oracle; argument errors and injected faults return their status without
touching a GPU.
"""
import ctypes
import os

import pytest

import oracle
from sparse_head_self_gb300 import _native, api
from sparse_head_self_gb300.build import build_all
from sparse_head_self_gb300.inputs import WORKLOADS


@pytest.fixture(scope="module", autouse=True)
def _built():
    build_all()
    yield


@pytest.mark.parametrize("checks", [False, True])
def test_exports_every_header_function(checks):
    # the library and its bounds-checked debug build (both made by build())
    from sparse_head_self_gb300.build import LIB, LIB_CHECKS
    names = _native.header_functions()
    assert "fibatt_fwd" in names and "fibatt_bwd" in names and "fibatt_support_build" in names
    L = ctypes.CDLL(LIB_CHECKS if checks else LIB)
    missing = [n for n in names if not hasattr(L, n)]
    assert not missing, missing
    assert set(names) == set(_native._SIGS), "ctypes signatures out of sync with the header"


def test_wythoff_rows_match_oracle():
    for i in range(1, 2001):
        assert api.wythoff_row(i) == oracle.wythoff_row(i)
    for i in (10**6, 10**7, 10**8):
        assert api.wythoff_row(i) == oracle.wythoff_row(i)


def test_wythoff_modified_rows_precede_row():
    for i in range(1, 300):
        a, b = api.wythoff_row(i)
        am, bm = api.wythoff_row_modified(i)
        # the modified pair continues into the row: am + bm = a and bm + a = b
        assert (am + bm, bm + a) == (a, b)
        assert oracle.fib_list(am, bm, b)[2:4] == [a, b]


def test_window_schedule_matches_oracle():
    for h, lo, hi in [(12, 5, 197), (12, 16, 1569), (16, 64, 16385), (3, 5, 65), (1, 4, 9), (7, 3, 3)]:
        assert api.window_schedule(h, lo, hi) == oracle.windows(h, lo, hi)


def _oracle_heads(wl, modified=False):
    w = oracle.windows(wl.H, wl.w_min, wl.w_max)
    heads = []
    for i in range(1, wl.H + 1):
        a, b = oracle.wythoff_row(i)
        if modified:
            a, b = 2 * a - b, b - a
        heads.append(oracle.Head.fibottention(a, b, w[i - 1], wl.diag))
    return heads


@pytest.mark.parametrize("name", list(WORKLOADS))
def test_support_tables_bit_exact(name):
    wl = WORKLOADS[name]
    sup = api.Support.wythoff(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag)
    got = sup.head_offsets()
    pairs = sup.pairs
    for h, head in enumerate(_oracle_heads(wl)):
        ref = oracle.signed_table(wl.N, head)
        assert got[h] == [int(x) for x in ref], (name, h)
        # |Omega_h| counted along the oracle's table: N - |delta| pairs per diagonal
        assert pairs[h] == sum(wl.N - abs(int(d)) for d in ref)
        if wl.N <= 400:
            assert pairs[h] == oracle.support_size(wl.N, head)


def test_tiny_pair_counts():
    wl = WORKLOADS["tiny"]
    sup = api.Support.wythoff(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag)
    assert sup.pairs == [563, 577, 515]


def test_modified_variant_tables_bit_exact():
    for name in ("tiny", "vitb", "video"):
        wl = WORKLOADS[name]
        sup = api.Support.wythoff(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag, modified=True)
        for h, head in enumerate(_oracle_heads(wl, modified=True)):
            assert sup.head_offsets()[h] == [int(x) for x in oracle.signed_table(wl.N, head)]


def test_distance_support_matches_oracle():
    N = 90
    dists = [[0, 3, 3, 9, 200], [5, 10, 15, 20, 25], list(range(N)), [1, 2, 4, 8, 16, 32, 64], []]
    for diag in (False, True):
        sup = api.Support.from_distances(N, dists, diag)
        for h, d in enumerate(dists):
            head = oracle.Head(d, N, diag)
            assert sup.head_offsets()[h] == [int(x) for x in oracle.signed_table(N, head)]
            assert sup.pairs[h] == oracle.support_size(N, head)


def test_global_token_pair_counts_match_oracle():
    for name in ("tiny", "vitb", "vitb_nodiag"):
        wl = WORKLOADS[name]
        sup = api.Support.wythoff(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag)
        banded = sup.pairs
        sup.set_global_token(True)
        heads = oracle.wythoff_heads(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag, global_token=True)
        assert sup.pairs == [oracle.support_size(wl.N, h) for h in heads]
        # the tables keep describing the banded part
        assert sup.head_offsets() == [[int(x) for x in oracle.signed_table(wl.N, h)] for h in heads]
        sup.set_global_token(False)
        assert sup.pairs == banded
    d = [[], [3, 9]]
    sup = api.Support.from_distances(12, d, False).set_global_token(True)
    assert sup.pairs == [oracle.support_size(12, oracle.Head(x, 12, False, global_token=True)) for x in d]


def test_global_token_unsupported_paths_fail_before_launch(monkeypatch):
    L = _native.lib()
    sup = api.Support.wythoff(3, 65, 5, 65, True).set_global_token(True)
    fake, lse = 1 << 20, 1 << 21   # never dereferenced: both calls fail their checks first
    monkeypatch.setenv("FIBATT_PATH", "generic")
    assert L.fibatt_fwd(sup.handle, 1, 64, 0, fake, fake, fake, 0.125, fake, lse, None) == 2
    assert "global" in L.fibatt_last_error().decode()
    assert L.fibatt_bwd_noalloc(sup.handle, 1, 64, 0, fake, fake, fake, fake, lse, fake, 0.1, fake, fake, fake,
                                None) == 2


def test_entry_limit_is_exact():
    # FIBATT_MAX_ENTRIES signed entries in total are accepted, one more is not
    L = _native.lib()
    h = ctypes.c_void_p()
    limit = 1024
    d = list(range(1, limit // 2 + 1))   # 512 distances -> 1024 signed entries without the diagonal
    assert L.fibatt_support_build_distances(1, 2000, api._i32([len(d)]), api._i32(d), 0, ctypes.byref(h)) == 0
    n, N, total = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    assert L.fibatt_support_info(h, ctypes.byref(n), ctypes.byref(N), ctypes.byref(total)) == 0
    assert total.value == limit
    L.fibatt_support_destroy(h)
    assert L.fibatt_support_build_distances(1, 2000, api._i32([len(d)]), api._i32(d), 1, ctypes.byref(h)) == 2
    assert "more than 1024 signed offsets" in L.fibatt_last_error().decode()


def test_permutation_reorders_heads():
    base = api.Support.wythoff(4, 100, 5, 100, True)
    perm = [2, 0, 3, 1]
    sup = api.Support.wythoff(4, 100, 5, 100, True, permutation=perm)
    b = base.head_offsets()
    assert sup.head_offsets() == [b[p] for p in perm]


def _status(fn, *args):
    return fn(*args)


def test_support_build_errors():
    L = _native.lib()
    h = ctypes.c_void_p()

    def build(H, N, a, b, w, diag=1):
        return L.fibatt_support_build(H, N, api._i64(a), api._i64(b), api._i64(w), diag, ctypes.byref(h))

    assert build(1, 10, [1], [2], [5]) == 0
    L.fibatt_support_destroy(h)
    assert build(0, 10, [1], [2], [5]) == 1
    assert build(1, 0, [1], [2], [5]) == 1
    assert build(1, 10, [-1], [2], [5]) == 1
    assert build(1, 10, [0], [0], [5]) == 1
    assert build(1, 10, [1], [2], [0]) == 1
    assert build(1, 10, [1], [2], [11]) == 1
    assert build(65, 10, [1] * 65, [2] * 65, [5] * 65) == 2
    assert "window" in L.fibatt_last_error().decode() or L.fibatt_last_error()
    # too many signed entries in total
    assert L.fibatt_support_build_distances(1, 2000, api._i32([1500]), api._i32(range(1500)), 0,
                                            ctypes.byref(h)) == 2
    assert L.fibatt_support_build_distances(1, 20, api._i32([1]), api._i32([-3]), 0,
                                            ctypes.byref(h)) == 1
    with pytest.raises(_native.FibattError):
        api.wythoff_row(0)
    with pytest.raises(_native.FibattError):
        api.window_schedule(3, 10, 5)


def test_fwd_argument_errors_without_launch(monkeypatch):
    L = _native.lib()
    # the generic backward takes a workspace, so its size check runs (and
    # fails) before anything could be launched with the fake pointers below
    monkeypatch.setenv("FIBATT_PATH", "generic")
    sup = api.Support.wythoff(3, 65, 5, 65, True)
    fake = 1 << 20  # never dereferenced: every case below fails its checks first
    lse = 1 << 21

    def fwd(B=1, D=64, dt=0, q=fake, o=fake, scale=0.125):
        return L.fibatt_fwd(sup.handle, B, D, dt, q, fake, fake, scale, o, lse, None)

    assert fwd(B=0) == 1
    assert fwd(D=32) == 2
    assert fwd(dt=7) == 2
    assert fwd(q=None) == 1
    assert fwd(q=fake + 8) == 1
    assert fwd(scale=float("inf")) == 1
    assert L.fibatt_fwd(None, 1, 64, 0, fake, fake, fake, 0.1, fake, lse, None) == 1
    ws = sup.bwd_workspace_bytes(2)
    # the larger of one fp32 per query row and the pair-weight scratch
    # (P and dS, max entries of one head x N fp32 each per (b, h))
    max_count = max(len(x) for x in sup.head_offsets())
    assert ws == ((max(2 * 3 * 65 * 4, 2 * 3 * 2 * max_count * 65 * 4) + 255) // 256) * 256
    # one byte short of what the generic backward touches (D_j, one fp32 per row)
    assert L.fibatt_bwd(sup.handle, 2, 64, 1, fake, fake, fake, fake, lse, fake, 0.1, fake, fake, fake,
                        fake, 2 * 3 * 65 * 4 - 1, None) == 1


def test_injected_faults_report_status(monkeypatch):
    L = _native.lib()
    sup = api.Support.wythoff(3, 65, 5, 65, True)
    fake, lse = 1 << 20, 1 << 21
    monkeypatch.setenv("FIBATT_FAULT", "launch")
    assert L.fibatt_fwd(sup.handle, 1, 64, 0, fake, fake, fake, 0.125, fake, lse, None) == 3
    assert "injected" in L.fibatt_last_error().decode()
    ws = sup.bwd_workspace_bytes(1)
    assert L.fibatt_bwd(sup.handle, 1, 64, 0, fake, fake, fake, fake, lse, fake, 0.1, fake, fake, fake,
                        fake, ws, None) == 3
    monkeypatch.setenv("FIBATT_FAULT", "arg")
    assert L.fibatt_fwd(sup.handle, 1, 64, 0, fake, fake, fake, 0.125, fake, lse, None) == 1
    with pytest.raises(_native.FibattError):
        _native.check(1)


def test_python_api_rejects_cpu_tensors():
    import torch
    sup = api.Support.wythoff(3, 65, 5, 65, True)
    q = torch.zeros(1, 3, 65, 64)
    with pytest.raises(ValueError, match="CUDA"):
        api.fwd(sup, q, q, q, 0.125)
