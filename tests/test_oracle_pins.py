"""Pins of the fp64 oracle against things other than itself.

Each test checks the oracle against a fact fixed by the Fibottention paper
(arXiv 2406.19391, Sec. 3) or the project README (Algorithms 1-3), or by
mathematics: printed values, closed forms, an independent construction of the
Wythoff array from Zeckendorf representations, dense library attention
(scipy / torch), and central finite differences.  None re-calls the oracle's
own routine to produce its expected value.
"""
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------ Wythoff array

def _zeckendorf(m: int) -> list[int]:
    """Indices i (F_2 = 1, F_3 = 2, F_4 = 3, ...) of m's Zeckendorf terms, greedy."""
    fibs = [0, 1, 1]  # F_0, F_1, F_2
    while fibs[-1] <= m:
        fibs.append(fibs[-1] + fibs[-2])
    idx = []
    i = len(fibs) - 1
    while m > 0:
        while fibs[i] > m:
            i -= 1
        idx.append(i)
        m -= fibs[i]
        i -= 2
    return idx, fibs


def _shift(m: int) -> int:
    """Zeckendorf successor: replace every term F_i of m by F_{i+1}."""
    idx, fibs = _zeckendorf(m)
    while len(fibs) <= max(idx) + 2:
        fibs.append(fibs[-1] + fibs[-2])
    return sum(fibs[i + 1] for i in idx)


def _wythoff_by_zeckendorf(rows: int):
    """Row n of the Wythoff array without the golden ratio: its first term is
    the n-th integer whose Zeckendorf sum contains F_2 = 1, and each later term
    shifts the previous one's representation up by one index."""
    out = []
    m = 0
    while len(out) < rows:
        m += 1
        idx, _ = _zeckendorf(m)
        if min(idx) == 2:
            a = m
            b = _shift(a)
            out.append((a, b, _shift(b), _shift(_shift(b))))
    return out


def test_wythoff_golden_rows():
    with open(os.path.join(GOLDEN, "wythoff_rows.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            row, terms = line.split(":")
            terms = [int(x) for x in terms.split()]
            a, b = oracle.wythoff_row(int(row))
            assert (a, b) == (terms[0], terms[1])
            assert oracle.fib_list(a, b, terms[-1])[: len(terms)] == terms


def test_wythoff_matches_zeckendorf_construction():
    ref = _wythoff_by_zeckendorf(400)
    for n, (a, b, c, d) in enumerate(ref, start=1):
        assert oracle.wythoff_row(n) == (a, b), n
        # the row continues by the Fibonacci recurrence (Algorithm 1)
        assert oracle.fib_list(a, b, d)[:4] == [a, b, c, d]


def test_wythoff_rows_partition_positive_integers():
    # Sec. 3.2: rows have no overlap and contain each positive integer once.
    M = 3000
    seen = np.zeros(M + 1, dtype=np.int64)
    n = 1
    while True:
        a, b = oracle.wythoff_row(n)
        if a > M:
            break
        for f in oracle.fib_list(a, b, M + 1):
            if f <= M:
                seen[f] += 1
        n += 1
    assert np.all(seen[1:] == 1)


def test_isqrt_and_floor_phi_large():
    for n in [0, 1, 2, 3, 4, 15, 16, 17, 10**12, 10**12 + 1, 2**61 - 1]:
        r = oracle.isqrt(n)
        assert r == math.isqrt(n)
    # floor(n*phi) against exact rational arithmetic on sqrt(5 n^2)
    for n in [1, 2, 3, 10, 1000, 123456789, 10**8]:
        assert oracle.floor_mul_phi(n) == (n + math.isqrt(5 * n * n)) // 2


# ----------------------------------------------------- Fibonacci (Alg. 1)

def _fib_std(n: int) -> int:
    """Standard Fibonacci F_n with F_{-1} = 1, F_0 = 0, F_1 = 1."""
    if n == -1:
        return 1
    x, y = 0, 1
    for _ in range(n):
        x, y = y, x + y
    return x


@pytest.mark.parametrize("a,b,w", [(1, 2, 65), (4, 7, 35), (6, 10, 1), (6, 10, 6),
                                   (0, 1, 20), (3, 3, 50), (40, 65, 16385), (5, 2, 100)])
def test_fib_list_closed_form_and_stop_rule(a, b, w):
    seq = oracle.fib_list(a, b, w)
    # term n (1-based) of Fib(a, b) is a*F_{n-2} + b*F_{n-1}
    for n, f in enumerate(seq, start=1):
        assert f == a * _fib_std(n - 2) + b * _fib_std(n - 1)
    # Algorithm 1 stops at the first term >= w (it always keeps a and b)
    assert len(seq) >= 2
    if len(seq) > 2:
        assert seq[-1] >= w and seq[-2] < w
    else:
        assert seq[1] >= w


def test_window_schedule_endpoints():
    # Sec. 3.2: w_1 = w_min, w_h = w_max, non-decreasing in between
    for h, lo, hi in [(12, 5, 197), (12, 16, 1569), (16, 64, 16385), (3, 5, 65), (2, 7, 7)]:
        w = oracle.windows(h, lo, hi)
        assert w[0] == lo and w[-1] == hi
        assert all(x <= y for x, y in zip(w, w[1:]))
    assert oracle.windows(3, 5, 65) == [5, 35, 65]   # tiny workload: 5 + 60*(i-1)/2
    assert oracle.windows(1, 9, 40) == [9]


# ------------------------------------------------------------ support set

def _closed_form_size(N, a, b, w, diag):
    # |Omega| = sum over distinct f in Fib(a,b) with 1 <= f <= min(w, N-1) of
    # 2 (N - f), plus N for the main diagonal (asked for, or 0 in Fib(a,b)).
    terms = set()
    n = 1
    while True:
        f = a * _fib_std(n - 2) + b * _fib_std(n - 1)
        terms.add(f)
        if n >= 2 and f >= w:
            break
        n += 1
    size = sum(2 * (N - f) for f in terms if 1 <= f <= min(w, N - 1))
    if diag or 0 in terms:
        size += N
    return size


def test_support_size_closed_form_random():
    rng = np.random.default_rng(1)
    for _ in range(150):
        N = int(rng.integers(1, 90))
        a = int(rng.integers(0, 12))
        b = int(rng.integers(0 if a else 1, 20))
        w = int(rng.integers(1, N + 1))
        diag = bool(rng.integers(0, 2))
        head = oracle.Head.fibottention(a, b, w, diag)
        assert oracle.support_size(N, head) == _closed_form_size(N, a, b, w, diag)


def test_tiny_workload_support_sizes():
    # N = 65, heads on Wythoff rows 1..3, w = 5, 35, 65, diagonal on:
    #   row 1, F = {1,2,3,5}:        2(64+63+62+60) + 65     = 563
    #   row 2, F = {4,7,11,18,29}:   2(61+58+54+47+36) + 65  = 577
    #   row 3, F = {6,10,16,26,42}:  2(59+55+49+39+23) + 65  = 515
    heads = oracle.wythoff_heads(3, 65, 5, 65, True)
    assert [oracle.support_size(65, h) for h in heads] == [563, 577, 515]


def test_support_is_symmetric_banded_toeplitz():
    for (a, b, w, diag, N) in [(1, 2, 5, True, 40), (4, 7, 30, False, 50), (0, 1, 9, False, 20)]:
        head = oracle.Head.fibottention(a, b, w, diag)
        M = oracle.support_mask(N, head)
        assert np.array_equal(M, M.T)
        for d in range(-(N - 1), N):
            diagv = np.diagonal(M, d)
            assert diagv.min() == diagv.max()          # depends on k - j only
        assert not M[np.abs(np.subtract.outer(np.arange(N), np.arange(N))) > w].any()


def test_signed_table_equals_mask_diagonals():
    for (a, b, w, diag, N) in [(1, 2, 5, True, 65), (6, 10, 65, True, 65), (4, 7, 35, False, 65),
                               (40, 65, 2000, True, 300), (0, 1, 12, False, 30)]:
        head = oracle.Head.fibottention(a, b, w, diag)
        M = oracle.support_mask(N, head)
        present = [d for d in range(-(N - 1), N) if np.diagonal(M, d).any()]
        assert list(oracle.signed_table(N, head)) == present


# ------------------------------------------------------------ forward pass

def _dense_ref(Q, K, V, scale, mask=None):
    S = scale * (Q @ K.T)
    if mask is not None:
        S = np.where(mask.astype(bool), S, -np.inf)
    P = scipy.special.softmax(S, axis=1)
    return P @ V, scipy.special.logsumexp(S, axis=1)


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_fwd_dense_equivalence():
    # With every distance 0..N-1 in the support, Fibottention is plain softmax
    # attention (scores scaled, row softmax, weighted sum of V).
    N, Dh = 37, 16
    Q, K, V = _rand((N, Dh), 0), _rand((N, Dh), 1), _rand((N, Dh), 2)
    head = oracle.Head(range(N), N, False)
    O, L = oracle.fwd_head(Q, K, V, head, 0.25)
    O_ref, L_ref = _dense_ref(Q, K, V, 0.25)
    np.testing.assert_allclose(O, O_ref, atol=1e-12, rtol=0)
    np.testing.assert_allclose(L, L_ref, atol=1e-12, rtol=0)


def test_fwd_matches_masked_library_softmax():
    N, Dh = 65, 8
    Q, K, V = _rand((N, Dh), 3), _rand((N, Dh), 4), _rand((N, Dh), 5)
    for head in oracle.wythoff_heads(3, N, 5, 65, True) + oracle.wythoff_heads(4, N, 7, 65, False):
        M = oracle.support_mask(N, head)
        rows = np.nonzero(M.any(axis=1))[0]
        O, L = oracle.fwd_head(Q, K, V, head, 0.125)
        O_ref, L_ref = _dense_ref(Q, K, V, 0.125, M)
        np.testing.assert_allclose(O[rows], O_ref[rows], atol=1e-12, rtol=0)
        np.testing.assert_allclose(L[rows], L_ref[rows], atol=1e-12, rtol=0)


def test_fwd_diagonal_only_is_identity_on_V():
    N, Dh = 23, 64
    Q, K, V = _rand((N, Dh), 6), _rand((N, Dh), 7), _rand((N, Dh), 8)
    head = oracle.Head([], N, True)
    O, L = oracle.fwd_head(Q, K, V, head, 0.125)
    assert np.array_equal(O, V)                       # single-term softmax weight is 1
    np.testing.assert_allclose(L, 0.125 * np.einsum("nd,nd->n", Q, K), atol=1e-13, rtol=0)


def test_fwd_empty_rows():
    # N = 3 with distances {4, 7}: no pair fits, every row is empty.
    N, Dh = 3, 8
    Q, K, V, dO = (_rand((N, Dh), s) for s in range(4))
    head = oracle.Head.fibottention(4, 7, 3, False)
    O, L = oracle.fwd_head(Q, K, V, head, 0.125)
    assert np.all(O == 0) and np.all(np.isneginf(L))
    dQ, dK, dV = oracle.bwd_head(Q, K, V, dO, head, 0.125)
    assert np.all(dQ == 0) and np.all(dK == 0) and np.all(dV == 0)


def test_fwd_row_subset_matches_full():
    N, Dh = 50, 8
    Q, K, V = _rand((N, Dh), 9), _rand((N, Dh), 10), _rand((N, Dh), 11)
    head = oracle.Head.fibottention(4, 7, 40, True)
    O, L = oracle.fwd_head(Q, K, V, head, 0.3)
    rows = [0, 7, 49, 21]
    Os, Ls = oracle.fwd_head(Q, K, V, head, 0.3, rows=rows)
    assert np.array_equal(Os, O[rows]) and np.array_equal(Ls, L[rows])


# ----------------------------------------------------------- backward pass

def _loss(Q, K, V, dO, head, scale):
    O, _ = oracle.fwd_head(Q, K, V, head, scale)
    return float(np.sum(O * dO))


def test_bwd_central_finite_differences():
    N, Dh, scale, h = 13, 4, 0.5, 1e-6
    Q, K, V, dO = (_rand((N, Dh), 20 + s) for s in range(4))
    for head in [oracle.Head.fibottention(1, 2, 5, True), oracle.Head.fibottention(4, 7, 12, False)]:
        dQ, dK, dV = oracle.bwd_head(Q, K, V, dO, head, scale)
        for X, G in [(Q, dQ), (K, dK), (V, dV)]:
            num = np.zeros_like(X)
            for idx in np.ndindex(*X.shape):
                old = X[idx]
                X[idx] = old + h
                lp = _loss(Q, K, V, dO, head, scale)
                X[idx] = old - h
                lm = _loss(Q, K, V, dO, head, scale)
                X[idx] = old
                num[idx] = (lp - lm) / (2 * h)
            np.testing.assert_allclose(G, num, atol=2e-7, rtol=0)


def test_bwd_matches_torch_autograd_masked_dense():
    N, Dh, scale = 40, 16, 0.125
    Q, K, V, dO = (_rand((N, Dh), 30 + s) for s in range(4))
    for head in oracle.wythoff_heads(3, N, 5, 40, True):
        M = torch.from_numpy(oracle.support_mask(N, head).astype(bool))
        q, k, v = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
        s = (scale * q @ k.T).masked_fill(~M, float("-inf"))
        o = torch.softmax(s, dim=1) @ v
        o.backward(torch.from_numpy(dO))
        dQ, dK, dV = oracle.bwd_head(Q, K, V, dO, head, scale)
        np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-12, rtol=0)


def test_bwd_row_subsets_match_full():
    N, Dh = 45, 8
    Q, K, V, dO = (_rand((N, Dh), 40 + s) for s in range(4))
    head = oracle.Head.fibottention(6, 10, 45, True)
    dQ, dK, dV = oracle.bwd_head(Q, K, V, dO, head, 0.2)
    qr, kr = [3, 44, 0], [10, 0, 44, 17]
    sQ, sK, sV = oracle.bwd_head(Q, K, V, dO, head, 0.2, qrows=qr, krows=kr)
    assert np.array_equal(sQ, dQ[qr]) and np.array_equal(sK, dK[kr]) and np.array_equal(sV, dV[kr])


def test_bwd_gradient_sums():
    # Softmax rows sum to one, so shifting every key by the same vector leaves
    # O unchanged: the rows of dK sum to zero within each head.
    N, Dh = 30, 8
    Q, K, V, dO = (_rand((N, Dh), 50 + s) for s in range(4))
    head = oracle.Head.fibottention(1, 2, 8, True)
    _, dK, _ = oracle.bwd_head(Q, K, V, dO, head, 0.4)
    np.testing.assert_allclose(dK.sum(axis=0), 0.0, atol=1e-12)


# ------------------------------------------------- global first token (CLS)
#
# README Algorithm 2 leaves row 0 and column 0 of its (N+1) x (N+1) mask all
# ones: the class token attends every key and every token attends it.

def _global_mask_by_definition(N, S, w, diag):
    """Omega by the set definition, plus row 0 and column 0 (numpy only)."""
    j = np.arange(N)[:, None]
    k = np.arange(N)[None, :]
    d = np.abs(j - k)
    M = np.isin(d, np.asarray(list(S), dtype=np.int64)) & (d <= w)
    if diag:
        M |= d == 0
    M[0, :] = True
    M[:, 0] = True
    return M


@pytest.mark.parametrize("N,S,w,diag", [(1, [1, 2], 5, False), (2, [], 2, False), (9, [1, 2, 3, 5, 8], 5, True),
                                        (40, [4, 7, 11, 18, 29], 30, False), (65, [6, 10, 16, 26, 42], 65, True)])
def test_global_token_support(N, S, w, diag):
    head = oracle.Head(S, w, diag, global_token=True)
    M = oracle.support_mask(N, head)
    assert np.array_equal(M.astype(bool), _global_mask_by_definition(N, S, w, diag))
    # closed form: the banded pairs, plus the 2N - 1 pairs of row/column 0,
    # minus those of row/column 0 that are banded already (c on each, the
    # diagonal pair (0, 0) counted once)
    c = sum(1 for f in set(S) if 1 <= f <= min(w, N - 1)) + (1 if diag or 0 in S else 0)
    base = oracle.support_size(N, oracle.Head(S, w, diag))
    assert oracle.support_size(N, head) == base + (2 * N - 1) - (2 * c - (1 if diag or 0 in S else 0))
    # the signed table describes the banded part only
    assert np.array_equal(oracle.signed_table(N, head), oracle.signed_table(N, oracle.Head(S, w, diag)))


def test_global_token_only_support():
    # no distances, no diagonal: query 0 is plain softmax attention over every
    # key, and every other query attends key 0 alone (its output is V_0)
    N, Dh, scale = 17, 8, 0.3
    Q, K, V = _rand((N, Dh), 60), _rand((N, Dh), 61), _rand((N, Dh), 62)
    head = oracle.Head([], N, False, global_token=True)
    O, L = oracle.fwd_head(Q, K, V, head, scale)
    O_ref, L_ref = _dense_ref(Q[:1], K, V, scale)
    np.testing.assert_allclose(O[0], O_ref[0], atol=1e-12, rtol=0)
    np.testing.assert_allclose(L[0], L_ref[0], atol=1e-12, rtol=0)
    assert np.array_equal(O[1:], np.broadcast_to(V[0], (N - 1, Dh)))
    np.testing.assert_allclose(L[1:], scale * Q[1:] @ K[0], atol=1e-13, rtol=0)


def test_global_token_fwd_bwd_match_torch_masked_dense():
    N, Dh, scale = 33, 16, 0.125
    Q, K, V, dO = (_rand((N, Dh), 70 + s) for s in range(4))
    for head in oracle.wythoff_heads(3, N, 5, 33, True, global_token=True) + \
            oracle.wythoff_heads(2, N, 4, 20, False, global_token=True):
        M = torch.from_numpy(_global_mask_by_definition(N, head.S, head.w, bool(head.diag)))
        q, k, v = (torch.tensor(x, requires_grad=True) for x in (Q, K, V))
        s = (scale * q @ k.T).masked_fill(~M, float("-inf"))
        o = torch.softmax(s, dim=1) @ v
        o.backward(torch.from_numpy(dO))
        O, L = oracle.fwd_head(Q, K, V, head, scale)
        np.testing.assert_allclose(O, o.detach().numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(L, torch.logsumexp(s, dim=1).detach().numpy(), atol=1e-12, rtol=0)
        dQ, dK, dV = oracle.bwd_head(Q, K, V, dO, head, scale)
        np.testing.assert_allclose(dQ, q.grad.numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(dK, k.grad.numpy(), atol=1e-12, rtol=0)
        np.testing.assert_allclose(dV, v.grad.numpy(), atol=1e-12, rtol=0)


def test_global_token_bwd_central_finite_differences():
    N, Dh, scale, h = 11, 4, 0.5, 1e-6
    Q, K, V, dO = (_rand((N, Dh), 80 + s) for s in range(4))
    head = oracle.Head.fibottention(4, 7, 9, False, global_token=True)
    dQ, dK, dV = oracle.bwd_head(Q, K, V, dO, head, scale)
    for X, G in [(Q, dQ), (K, dK), (V, dV)]:
        num = np.zeros_like(X)
        for idx in np.ndindex(*X.shape):
            old = X[idx]
            X[idx] = old + h
            lp = _loss(Q, K, V, dO, head, scale)
            X[idx] = old - h
            lm = _loss(Q, K, V, dO, head, scale)
            X[idx] = old
            num[idx] = (lp - lm) / (2 * h)
        np.testing.assert_allclose(G, num, atol=2e-7, rtol=0)
