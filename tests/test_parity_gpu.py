"""GPU parity: libfibatt (through the C ABI) against the fp64 oracle.

Small cases are compared element by element on every output; the full-size
workloads, in the same launch configuration as bench.py, are compared on
every output where the oracle is fast enough and on seeded row samples
(edges included) otherwise.  Tolerances are in tests/gpu_helpers.py.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import (assert_close, assert_close_global, band_edge_rows, make_inputs, oracle_heads,
                         pick_rows, support_for, to_dev)
from sparse_head_self_gb300 import api
from sparse_head_self_gb300.inputs import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

oracle.set_threads(oracle.max_threads())


@pytest.fixture
def kernel_path(request, monkeypatch):
    """Select the kernel family through FIBATT_PATH for one test: generic
    (global-memory kernels), resident (shared-memory staged), flat (the
    resident arithmetic on rows read from global memory; backward generic)
    or auto (the library's choice)."""
    path = getattr(request, "param", "auto")
    monkeypatch.delenv("FIBATT_STREAM", raising=False)
    monkeypatch.delenv("FIBATT_STREAM_WINDOW", raising=False)
    if path == "auto":
        monkeypatch.delenv("FIBATT_PATH", raising=False)
    elif path == "flat_legacy":   # the flat kernels that predate the streaming ones
        monkeypatch.setenv("FIBATT_PATH", "flat")
        monkeypatch.setenv("FIBATT_STREAM", "0")
    elif path == "flat_window":   # the streaming forward with the near window staged (on request)
        monkeypatch.setenv("FIBATT_PATH", "flat")
        monkeypatch.setenv("FIBATT_STREAM_WINDOW", "1")
    else:
        monkeypatch.setenv("FIBATT_PATH", path)
    return path


def _fwd_full(wl, seed=0):
    q, k, v, _ = make_inputs(wl, seed, with_grad=False)
    sup = support_for(wl)
    O, L = api.fwd(sup, *to_dev(q, k, v), wl.scale)
    O_ref, L_ref = oracle.fwd(q, k, v, oracle_heads(wl), wl.scale)
    assert_close(f"{wl.name} O", O.float().cpu(), O_ref, wl.dtype)
    assert_close(f"{wl.name} LSE", L.cpu(), L_ref, wl.dtype, lse=True)


def _bwd_full(wl, seed=0):
    q, k, v, do = make_inputs(wl, seed)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    rQ, rK, rV = oracle.bwd(q, k, v, do, oracle_heads(wl), wl.scale)
    assert_close(f"{wl.name} dQ", dQ.float().cpu(), rQ, wl.dtype)
    assert_close(f"{wl.name} dK", dK.float().cpu(), rK, wl.dtype)
    assert_close(f"{wl.name} dV", dV.float().cpu(), rV, wl.dtype)


# ------------------------------------------------------------ small, full

@pytest.mark.parametrize("kernel_path", ["generic", "resident", "flat", "flat_legacy"], indirect=True)
def test_tiny_fwd_fp32_full(kernel_path):
    _fwd_full(WORKLOADS["tiny"])


@pytest.mark.parametrize("kernel_path", ["generic", "resident", "flat", "flat_legacy"], indirect=True)
def test_tiny_bwd_fp32_full(kernel_path):
    _bwd_full(WORKLOADS["tiny"])


@pytest.mark.parametrize("kernel_path", ["generic", "resident", "flat"], indirect=True)
@pytest.mark.parametrize("name", ["vitb", "vitb_nodiag"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_vitb_shape_small_batch_full(name, dtype, kernel_path):
    wl = Workload(**{**WORKLOADS[name].__dict__, "B": 2, "dtype": dtype})
    _fwd_full(wl, seed=5)
    _bwd_full(wl, seed=5)


def test_video_shape_one_batch_fwd_full():
    wl = WORKLOADS["video"].with_batch(1)
    _fwd_full(wl, seed=7)


@pytest.mark.parametrize("key_unroll", ["1", "2"])
def test_video_shape_two_heads_bwd_key_pass_steps(key_unroll, monkeypatch):
    # the streaming key pass with one or two table entries per step (ragged
    # tails of odd entry counts included: heads with 13 and 19 entries)
    monkeypatch.setenv("FIBATT_PATH", "flat")
    monkeypatch.setenv("FIBATT_KEY_UNROLL", key_unroll)
    wl = WORKLOADS["video"].with_batch(1)
    q, k, v, do = make_inputs(wl, 10)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    heads = oracle_heads(wl)
    for h in (0, 1, wl.H - 1):
        rQ, rK, rV = oracle.bwd_head(q[0, h], k[0, h], v[0, h], do[0, h], heads[h], wl.scale)
        assert_close(f"video h{h} dQ", dQ[0, h].float().cpu(), rQ, wl.dtype)
        assert_close(f"video h{h} dK", dK[0, h].float().cpu(), rK, wl.dtype)
        assert_close(f"video h{h} dV", dV[0, h].float().cpu(), rV, wl.dtype)


@pytest.mark.parametrize("kernel_path", ["generic", "flat", "flat_window", "flat_legacy"], indirect=True)
def test_video_shape_two_heads_bwd_full(kernel_path):
    # every row of two heads (the narrowest and the widest window) of one
    # batch element: every gradient compared with the oracle's
    wl = WORKLOADS["video"].with_batch(1)
    q, k, v, do = make_inputs(wl, 9)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    heads = oracle_heads(wl)
    for h in (0, wl.H - 1):
        rQ, rK, rV = oracle.bwd_head(q[0, h], k[0, h], v[0, h], do[0, h], heads[h], wl.scale)
        assert_close(f"video h{h} dQ", dQ[0, h].float().cpu(), rQ, wl.dtype)
        assert_close(f"video h{h} dK", dK[0, h].float().cpu(), rK, wl.dtype)
        assert_close(f"video h{h} dV", dV[0, h].float().cpu(), rV, wl.dtype)


@pytest.mark.parametrize("kernel_path", ["generic", "flat", "flat_legacy", "auto"], indirect=True)
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 63, 64, 65, 127, 129, 300])
@pytest.mark.parametrize("diag", [False, True])
def test_edge_sizes(N, diag, kernel_path):
    # rows 1..4 of the Wythoff array with windows up to N: includes heads whose
    # whole support is empty (N <= a_h without the diagonal)
    H = 4
    wl = Workload("edge", 2, H, N, 64, "f32", 1, N, diag, True)
    _fwd_full(wl, seed=N)
    _bwd_full(wl, seed=N)


@pytest.mark.parametrize("shape", ["0", "1"])
@pytest.mark.parametrize("N", [1, 5, 63, 64, 65, 81, 200, 300, 1569])
def test_window_forward_bf16(N, shape, monkeypatch):
    # the streaming forward that stages the key and value rows of the near
    # table entries (|offset| up to 88 or 96) in shared memory (a variant
    # taken on request; the plain streaming forward is faster): six Wythoff
    # heads (near entries only, near and far, far only) and three heads of
    # every distance below 170 (near and far entries side by side; the whole
    # table stays within the 1024-entry limit), every output against the
    # oracle; block edges at 64 and 80 rows, windows clipped at both ends of
    # the sequence
    monkeypatch.setenv("FIBATT_PATH", "flat")
    monkeypatch.delenv("FIBATT_STREAM", raising=False)
    monkeypatch.setenv("FIBATT_STREAM_WINDOW", "1")
    monkeypatch.setenv("FIBATT_WINDOW_SHAPE", shape)
    wl = Workload("window", 2, 6, N, 64, "bf16", 1, N, True, True)
    _fwd_full(wl, seed=N + 11)
    wl = Workload("window_dense", 2, 3, N, 64, "bf16", 1, N, True, True)
    q, k, v, _ = make_inputs(wl, N + 12, with_grad=False)
    dist = list(range(min(N, 170)))
    sup = api.Support.from_distances(N, [dist] * wl.H, True)
    O, L = api.fwd(sup, *to_dev(q, k, v), wl.scale)
    O_ref, L_ref = oracle.fwd(q, k, v, [oracle.Head(dist, N, True)] * wl.H, wl.scale)
    assert_close("window dense O", O.float().cpu(), O_ref, "bf16")
    assert_close("window dense LSE", L.cpu(), L_ref, "bf16", lse=True)


def _offset_view(t, elems):
    """A copy of t placed `elems` elements into a larger buffer: 16-byte but
    not 32-byte aligned when elems x element size is 16 (mod 32)."""
    buf = torch.empty(t.numel() + elems, dtype=t.dtype, device=t.device)
    v = buf[elems:].view(t.shape)
    v.copy_(t)
    return v


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_flat_rows_sixteen_byte_aligned(dtype, monkeypatch):
    # the streaming kernels read 32-byte pieces of rows; tensors that are
    # only 16-byte aligned (the boundary's requirement) take the older flat
    # kernels, with the same results
    monkeypatch.setenv("FIBATT_PATH", "flat")
    monkeypatch.delenv("FIBATT_STREAM", raising=False)
    wl = Workload("edge", 2, 4, 129, 64, dtype, 1, 129, True, True)
    q, k, v, do = make_inputs(wl, 5)
    elems = 16 // (4 if dtype == "f32" else 2)
    qd, kd, vd, dod = (_offset_view(t.cuda(), elems) for t in (q, k, v, do))
    assert all(t.data_ptr() % 32 == 16 for t in (qd, kd, vd, dod))
    sup = support_for(wl)
    O = _offset_view(torch.zeros_like(qd), elems)
    L = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    api.fwd(sup, qd, kd, vd, wl.scale, O=O, LSE=L)
    heads = oracle_heads(wl)
    O_ref, L_ref = oracle.fwd(q, k, v, heads, wl.scale)
    assert_close("O", O.float().cpu(), O_ref, wl.dtype)
    assert_close("LSE", L.cpu(), L_ref, wl.dtype, lse=True)
    dQ, dK, dV = (_offset_view(torch.zeros_like(qd), elems) for _ in range(3))
    api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale, dQ=dQ, dK=dK, dV=dV)
    rQ, rK, rV = oracle.bwd(q, k, v, do, heads, wl.scale)
    assert_close("dQ", dQ.float().cpu(), rQ, wl.dtype)
    assert_close("dK", dK.float().cpu(), rK, wl.dtype)
    assert_close("dV", dV.float().cpu(), rV, wl.dtype)


@pytest.mark.parametrize("qsplit", ["1", "2", "3", "7", "40"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_resident_query_chunks(qsplit, dtype, monkeypatch):
    # every split of the 197 queries into chunks, ragged last chunk included
    monkeypatch.setenv("FIBATT_PATH", "resident")
    monkeypatch.setenv("FIBATT_QSPLIT", qsplit)
    wl = Workload(**{**WORKLOADS["vitb"].__dict__, "B": 2, "dtype": dtype})
    _fwd_full(wl, seed=23)


@pytest.mark.parametrize("snake", ["0", "1"])
@pytest.mark.parametrize("split", ["0", "1"])
def test_resident_last_wave_pieces(split, snake, monkeypatch):
    # with the split: 7 x 12 heads x 2 chunks = 168 units on (at most) 152
    # CTAs, the units of the partial last wave cut into one-round pieces, some
    # of them past the end of their chunk (empty); without: 20 x 24 = 480
    # units, three full waves, the second of them reversed by the snake order
    monkeypatch.setenv("FIBATT_PATH", "resident")
    monkeypatch.setenv("FIBATT_QSPLIT", "2")
    monkeypatch.setenv("FIBATT_SPLIT_TAIL", split)
    monkeypatch.setenv("FIBATT_FWD_SNAKE", snake)
    wl = WORKLOADS["vitb"].with_batch(7 if split == "1" else 20)
    _fwd_full(wl, seed=13)


@pytest.mark.parametrize("mode", ["0", "1", "2"])
@pytest.mark.parametrize("B", [13, 38])
def test_resident_first_unit_alone(mode, B, monkeypatch):
    # a CTA's second unit copied only after its first unit landed (1: the
    # forward, the default; 2: both kernels; 0: neither), every output and
    # gradient; B = 13: a last wave of pieces, B = 38: three whole waves
    monkeypatch.setenv("FIBATT_PATH", "resident")
    monkeypatch.setenv("FIBATT_FIRST_ALONE", mode)
    wl = WORKLOADS["vitb"].with_batch(B)
    _fwd_full(wl, seed=41 + B)
    _bwd_full(wl, seed=41 + B)


@pytest.mark.parametrize("gwarps", ["12", "11", "7"])
@pytest.mark.parametrize("B", [13, 20])
def test_resident_forward_rounds_circulate(gwarps, B, monkeypatch):
    # fewer consumer warps than the 13 rounds of a 197-row head: the rounds
    # circulate over the warps from unit to unit (B = 13: a last wave cut
    # into pieces; B = 20: 240 whole-head units, two waves), every output
    monkeypatch.setenv("FIBATT_PATH", "resident")
    monkeypatch.setenv("FIBATT_FWD_GWARPS", gwarps)
    _fwd_full(WORKLOADS["vitb"].with_batch(B), seed=31 + B)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("pieces", ["0", "1", "1-serial"])
@pytest.mark.parametrize("B", [13, 14, 15, 27])
def test_resident_bwd_last_wave_pieces(B, pieces, dtype, monkeypatch):
    # 156, 168, 180 or 324 heads on (at most) 152 CTAs: the 4, 16, 28 or 20
    # heads of the partial last wave are cut into pieces of one, two or three
    # rounds (fp32: more), each piece recomputing P and dS for its key rows
    # (B = 27: two full waves, the second in snake order); every gradient of
    # every head compared with the oracle
    # one-round pieces run spread over nine warps, or ("1-serial") on two
    monkeypatch.setenv("FIBATT_PATH", "resident")
    monkeypatch.setenv("FIBATT_BWD_PIECES", pieces[0])
    monkeypatch.setenv("FIBATT_BWD_PIECE_PAR", "0" if pieces.endswith("serial") else "1")
    # fp32 rows: four lanes per row, 25 rounds of 8 rows, one stage
    _bwd_full(Workload(**{**WORKLOADS["vitb"].__dict__, "B": B, "dtype": dtype}), seed=B)


@pytest.mark.parametrize("kernel_path", ["generic", "resident", "flat"], indirect=True)
@pytest.mark.parametrize("scale", [0.0, 1e-3, -0.5, 3.0])
def test_extreme_scales(scale, kernel_path):
    # uniform weights (scale 0), nearly uniform, negative, and peaked
    # softmaxes (the running maximum is raised many times) in fp32
    wl = Workload(**{**WORKLOADS["vitb"].__dict__, "B": 1, "dtype": "f32", "scale": scale})
    q, k, v, do = make_inputs(wl, 31)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, scale)
    heads = oracle_heads(wl)
    O_r, L_r = oracle.fwd(q, k, v, heads, scale)
    rQ, rK, rV = oracle.bwd(q, k, v, do, heads, scale)
    # the peaked case has scores up to ~40 (natural units): compare relative to the magnitudes
    tol = 1e-5 * max(1.0, abs(scale) * 8)
    for n, g, r in (("O", O, O_r), ("LSE", L, L_r), ("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        d = np.abs(g.double().cpu().numpy() - r)
        assert d.max() <= tol * max(1.0, float(np.abs(r).max())), f"{n} scale {scale}: {d.max():.3e}"


@pytest.mark.parametrize("kernel_path", ["generic", "resident", "flat"], indirect=True)
def test_empty_support_rows_are_zero(kernel_path):
    # N = 3, row 2 of the Wythoff array (4, 7), no diagonal: no pair at all
    N = 3
    sup = api.Support.build(N, [4], [7], [3], False)
    q, k, v, do = (torch.randn(1, 1, N, 64, device="cuda") for _ in range(4))
    O, L = api.fwd(sup, q, k, v, 0.125)
    assert torch.all(O == 0) and torch.all(torch.isneginf(L))
    dQ, dK, dV = api.bwd(sup, q, k, v, O, L, do, 0.125)
    assert torch.all(dQ == 0) and torch.all(dK == 0) and torch.all(dV == 0)


@pytest.mark.parametrize("kernel_path", ["generic", "resident", "flat"], indirect=True)
def test_diagonal_only_support_returns_V(kernel_path):
    N = 77
    sup = api.Support.from_distances(N, [[], []], True)
    g = torch.Generator(device="cuda").manual_seed(3)
    q, k, v = (torch.randn(3, 2, N, 64, device="cuda", generator=g) for _ in range(3))
    O, L = api.fwd(sup, q, k, v, 0.125)
    assert torch.equal(O, v)      # a single-term softmax has weight exactly 1
    ref = 0.125 * (q.double() * k.double()).sum(-1)
    assert (L.double() - ref).abs().max().item() <= 1e-5


@pytest.mark.parametrize("kernel_path", ["generic", "flat", "auto"], indirect=True)
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_dense_support_equals_softmax_attention(dtype, kernel_path):
    # every distance 0..N-1: plain softmax attention (checked against the oracle,
    # itself pinned to library softmax attention)
    N, H = 150, 2
    wl = Workload("dense", 2, H, N, 64, dtype, 1, N, True, True)
    q, k, v, do = make_inputs(wl, 11)
    sup = api.Support.from_distances(N, [list(range(N))] * H, True)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    heads = [oracle.Head(range(N), N, True)] * H
    O_ref, L_ref = oracle.fwd(q, k, v, heads, wl.scale)
    assert_close("dense O", O.float().cpu(), O_ref, dtype)
    assert_close("dense LSE", L.cpu(), L_ref, dtype, lse=True)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    rQ, rK, rV = oracle.bwd(q, k, v, do, heads, wl.scale)
    for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        assert_close(f"dense {n}", g.float().cpu(), r, dtype)


@pytest.mark.parametrize("kernel_path", ["generic", "flat", "auto"], indirect=True)
def test_modified_wythoff_variant(kernel_path):
    wl = WORKLOADS["tiny"]
    q, k, v, do = make_inputs(wl, 13)
    sup = support_for(wl, modified=True)
    heads = oracle_heads(wl, modified=True)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    O_ref, L_ref = oracle.fwd(q, k, v, heads, wl.scale)
    assert_close("mod O", O.cpu(), O_ref, "f32")
    assert_close("mod LSE", L.cpu(), L_ref, "f32", lse=True)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    rQ, rK, rV = oracle.bwd(q, k, v, do, heads, wl.scale)
    for n, g, r in (("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        assert_close(f"mod {n}", g.cpu(), r, "f32")


def test_autograd_function_matches_direct_calls():
    wl = WORKLOADS["tiny"]
    q, k, v, do = make_inputs(wl, 17)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    leaves = [t.clone().requires_grad_(True) for t in (qd, kd, vd)]
    out = api.fibottention(*leaves, sup, wl.scale)
    out.backward(dod)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    assert torch.equal(out, O)
    for g, r in zip((leaves[0].grad, leaves[1].grad, leaves[2].grad), (dQ, dK, dV)):
        assert torch.equal(g, r)


def test_side_stream_and_repeatability():
    wl = WORKLOADS["vitb"].with_batch(3)
    q, k, v, _ = make_inputs(wl, 19, with_grad=False)
    sup = support_for(wl)
    qd, kd, vd = to_dev(q, k, v)
    O1, L1 = api.fwd(sup, qd, kd, vd, wl.scale)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        O2, L2 = api.fwd(sup, qd, kd, vd, wl.scale, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    assert torch.equal(O1, O2) and torch.equal(L1, L2)


@pytest.mark.parametrize("kernel_path", ["generic", "flat", "auto"], indirect=True)
def test_chained_calls_match_synchronised_calls(kernel_path):
    """Launches are programmatic dependent launches: each kernel may start
    while the previous one drains.  A chain that reuses its buffers (fwd
    writes O while the previous bwd still reads it, and so on) must give
    what the same calls give with a synchronisation between each."""
    wl = WORKLOADS["vitb"].with_batch(4)
    sup = support_for(wl)
    inputs = [to_dev(*make_inputs(wl, 60 + i)) for i in range(3)]
    ref = []
    for qd, kd, vd, dod in inputs:
        O, L = api.fwd(sup, qd, kd, vd, wl.scale)
        torch.cuda.synchronize()
        dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
        torch.cuda.synchronize()
        ref.append([t.clone() for t in (O, L, dQ, dK, dV)])
    # one O / LSE for the whole chain (the next fwd overwrites what the
    # previous bwd reads); gradients of each call kept apart
    O = torch.empty_like(inputs[0][0])
    L = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    grads = [[torch.empty_like(O) for _ in range(3)] for _ in range(6)]
    for i in range(6):
        qd, kd, vd, dod = inputs[i % 3]
        api.fwd(sup, qd, kd, vd, wl.scale, O=O, LSE=L)
        api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale, dQ=grads[i][0], dK=grads[i][1], dV=grads[i][2])
    torch.cuda.synchronize()
    assert torch.equal(O, ref[2][0]) and torch.equal(L, ref[2][1])
    for i in range(6):
        for a, b in zip(grads[i], ref[i % 3][2:]):
            assert torch.equal(a, b)


# ------------------------------------------------- global first token (CLS)

def _global_fwd_bwd(wl, seed, heads_subset=None):
    q, k, v, do = make_inputs(wl, seed)
    sup = support_for(wl, global_token=True)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    torch.cuda.synchronize()
    heads = oracle_heads(wl, global_token=True)
    hs = range(wl.H) if heads_subset is None else heads_subset
    for b in range(wl.B):
        for h in hs:
            Or, Lr = oracle.fwd_head(q[b, h], k[b, h], v[b, h], heads[h], wl.scale)
            assert_close_global(f"O b{b} h{h}", O[b, h].float().cpu(), Or, wl.dtype)
            assert_close_global(f"LSE b{b} h{h}", L[b, h].cpu(), Lr, wl.dtype, lse=True)
            rQ, rK, rV = oracle.bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], heads[h], wl.scale)
            assert_close_global(f"dQ b{b} h{h}", dQ[b, h].float().cpu(), rQ, wl.dtype)
            assert_close_global(f"dK b{b} h{h}", dK[b, h].float().cpu(), rK, wl.dtype)
            assert_close_global(f"dV b{b} h{h}", dV[b, h].float().cpu(), rV, wl.dtype)


@pytest.mark.parametrize("kernel_path", ["resident", "flat", "flat_legacy"], indirect=True)
def test_global_token_tiny_fp32(kernel_path):
    _global_fwd_bwd(WORKLOADS["tiny"], 21)


@pytest.mark.parametrize("kernel_path", ["resident", "flat"], indirect=True)
@pytest.mark.parametrize("name", ["vitb", "vitb_nodiag"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_global_token_vitb_shape(name, dtype, kernel_path):
    _global_fwd_bwd(Workload(**{**WORKLOADS[name].__dict__, "B": 2, "dtype": dtype}), 22)


@pytest.mark.parametrize("kernel_path", ["resident", "flat", "flat_legacy", "auto"], indirect=True)
@pytest.mark.parametrize("N", [1, 2, 3, 9, 40])
def test_global_token_edge_sizes(N, kernel_path):
    wl = Workload("edge", 2, 3, N, 64, "f32", 1, N, False, True)
    _global_fwd_bwd(wl, 23)


@pytest.mark.parametrize("fuse", ["1", "0", None])
@pytest.mark.parametrize("name,dtype,B", [("vitb", "bf16", 13), ("vitb", "f32", 13), ("vitb_nodiag", "bf16", 13),
                                          ("vitb", "bf16", 38)])
def test_global_token_whole_heads(name, dtype, B, fuse, monkeypatch):
    # B H >= the SM count: whole-head units, where row 0 is computed inside
    # the resident forward (fuse 1, the default) or by the dense row kernel
    # (fuse 0).  B = 13 leaves 4 units for the last wave, cut into pieces:
    # the piece holding query 0 stages its whole head and computes row 0;
    # B = 38 fills whole waves
    monkeypatch.delenv("FIBATT_PATH", raising=False)
    if fuse is None:
        monkeypatch.delenv("FIBATT_GT_FUSE", raising=False)
    else:
        monkeypatch.setenv("FIBATT_GT_FUSE", fuse)
    _global_fwd_bwd(Workload(**{**WORKLOADS[name].__dict__, "B": B, "dtype": dtype}), 25)


@pytest.mark.parametrize("fuse", ["1", "0"])
def test_global_token_vitb_batch_64(fuse, monkeypatch):
    # the bench's ViT-B shape (768 heads: five waves and a last wave of 8
    # units, cut into pieces), heads 0, 5 and 11 of every batch element
    monkeypatch.delenv("FIBATT_PATH", raising=False)
    monkeypatch.setenv("FIBATT_GT_FUSE", fuse)
    wl = Workload(**{**WORKLOADS["vitb"].__dict__, "B": 64})
    _global_fwd_bwd(wl, 27, heads_subset=(0, 5, wl.H - 1))


def test_global_token_many_waves():
    # B = 104 (1248 whole-head units, 8.2 waves with a last wave of 32): row 0
    # computed inside the resident forward because of the number of waves;
    # heads 0 and 11 of every batch element compared
    wl = Workload(**{**WORKLOADS["vitb"].__dict__, "B": 104})
    _global_fwd_bwd(wl, 26, heads_subset=(0, wl.H - 1))


@pytest.mark.parametrize("fuse", ["1", "0"])
@pytest.mark.parametrize("N", [1, 2, 9, 40])
def test_global_token_whole_heads_edge_sizes(N, fuse, monkeypatch):
    # short heads, 180 of them: many stages; N = 1 has empty tables (no
    # fusion then, the row kernel writes row 0)
    monkeypatch.delenv("FIBATT_PATH", raising=False)
    monkeypatch.setenv("FIBATT_GT_FUSE", fuse)
    _global_fwd_bwd(Workload("edge", 60, 3, N, 64, "f32", 1, N, False, True), 26)


@pytest.mark.parametrize("cluster", ["1", "3", None])
def test_global_token_video_two_heads(cluster, monkeypatch):
    # the dense row and column of token 0 split over clusters of 1, 3 or (the
    # library's choice) 8 CTAs per head
    if cluster is None:
        monkeypatch.delenv("FIBATT_GT_CLUSTER", raising=False)
    else:
        monkeypatch.setenv("FIBATT_GT_CLUSTER", cluster)
    wl = WORKLOADS["video"].with_batch(1)
    _global_fwd_bwd(wl, 24, heads_subset=(0, wl.H - 1))


@pytest.mark.parametrize("kernel_path", ["flat", "flat_legacy"], indirect=True)
def test_global_token_long_rows(kernel_path):
    # 5000 tokens: beyond the length at which the streaming forward computes
    # the dense row 0 in its own grid, so the dense row kernel takes it
    wl = Workload("gt_long", 1, 2, 5000, 64, "bf16", 64, 5000, True, True)
    _global_fwd_bwd(wl, 25)


def test_global_token_only_support_gives_v0():
    # no distances, no diagonal: every query but token 0 attends key 0 alone
    N, B = 50, 2
    sup = api.Support.from_distances(N, [[], []], False).set_global_token(True)
    wl = Workload("g", B, 2, N, 64, "f32", 2, 2, False, True)
    q, k, v, _ = make_inputs(wl, 25, with_grad=False)
    O, L = api.fwd(sup, *to_dev(q, k, v), wl.scale)
    torch.cuda.synchronize()
    assert torch.equal(O[:, :, 1:].cpu(), v[:, :, :1].expand(B, 2, N - 1, 64))


@pytest.mark.parametrize("name", ["vitb", "video"])
def test_cuda_graph_capture_replays_the_step(name):
    # the support travels as a kernel argument and the calls neither allocate
    # nor synchronise, so fwd + bwd can be captured once and replayed; the
    # first (eager) call sets up the plans before the capture
    wl = WORKLOADS[name].with_batch(2)
    sup = support_for(wl)
    q, k, v, do = make_inputs(wl, 41)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O = torch.empty_like(qd)
    L = torch.empty((wl.B, wl.H, wl.N), dtype=torch.float32, device="cuda")
    dQ, dK, dV = (torch.empty_like(qd) for _ in range(3))
    ws = torch.empty(sup.bwd_workspace_bytes(wl.B), dtype=torch.uint8, device="cuda")

    def step():
        api.fwd(sup, qd, kd, vd, wl.scale, O=O, LSE=L)
        api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale, dQ=dQ, dK=dK, dV=dV, workspace=ws)

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (O, L, dQ, dK, dV)]
    g = torch.cuda.CUDAGraph()
    for t in (O, L, dQ, dK, dV):
        t.zero_()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip((O, L, dQ, dK, dV), ref):
        assert torch.equal(a, b)


# ----------------------------------------------- full sizes, bench launches

@pytest.mark.parametrize("name", ["vitb", "vitb_nodiag"])
def test_vitb_full_size_fwd_all_outputs(name):
    _fwd_full(WORKLOADS[name])


def test_no_device_error_recorded():
    import ctypes
    from sparse_head_self_gb300 import _native
    code = ctypes.c_uint(123)
    _native.check(_native.lib().fibatt_device_error(1, ctypes.byref(code)))
    assert code.value == 0


def _sampled(wl, nbh, nrows, seed, backward):
    q, k, v, do = make_inputs(wl, 0, with_grad=backward)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    if backward:
        dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    torch.cuda.synchronize()
    heads = oracle_heads(wl)
    rng = np.random.default_rng(seed)
    picks = {(0, 0), (wl.B - 1, wl.H - 1)}
    while len(picks) < nbh:
        picks.add((int(rng.integers(wl.B)), int(rng.integers(wl.H))))
    for (b, h) in sorted(picks):
        rows = pick_rows(wl.N, nrows, seed + 31 * b + h)
        Or, Lr = oracle.fwd_head(q[b, h], k[b, h], v[b, h], heads[h], wl.scale, rows=rows)
        assert_close(f"{wl.name} O[{b},{h}]", O[b, h, rows].float().cpu(), Or, wl.dtype)
        assert_close(f"{wl.name} LSE[{b},{h}]", L[b, h, rows].cpu(), Lr, wl.dtype, lse=True)
        if backward:
            rQ, rK, rV = oracle.bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], heads[h], wl.scale,
                                         qrows=rows, krows=rows)
            assert_close(f"{wl.name} dQ[{b},{h}]", dQ[b, h, rows].float().cpu(), rQ, wl.dtype)
            assert_close(f"{wl.name} dK[{b},{h}]", dK[b, h, rows].float().cpu(), rK, wl.dtype)
            assert_close(f"{wl.name} dV[{b},{h}]", dV[b, h, rows].float().cpu(), rV, wl.dtype)


def _every_head_band_edges(wl, nrows, seed):
    """Every (b, h) head of the workload at full size, in the bench's launch
    configuration: forward and backward outputs on each head's band-edge rows
    (band_edge_rows) plus a seeded sample, element by element."""
    q, k, v, do = make_inputs(wl, 0)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    torch.cuda.synchronize()
    O, L, dQ, dK, dV = (x.float().cpu() for x in (O, L, dQ, dK, dV))
    heads = oracle_heads(wl)
    w = oracle.windows(wl.H, wl.w_min, wl.w_max)
    for h in range(wl.H):
        rows = band_edge_rows(wl.N, heads[h], w[h], nrows, seed + h)
        for b in range(wl.B):
            Or, Lr = oracle.fwd_head(q[b, h], k[b, h], v[b, h], heads[h], wl.scale, rows=rows)
            rQ, rK, rV = oracle.bwd_head(q[b, h], k[b, h], v[b, h], do[b, h], heads[h], wl.scale,
                                         qrows=rows, krows=rows)
            assert_close(f"{wl.name} O[{b},{h}]", O[b, h, rows], Or, wl.dtype)
            assert_close(f"{wl.name} LSE[{b},{h}]", L[b, h, rows], Lr, wl.dtype, lse=True)
            assert_close(f"{wl.name} dQ[{b},{h}]", dQ[b, h, rows], rQ, wl.dtype)
            assert_close(f"{wl.name} dK[{b},{h}]", dK[b, h, rows], rK, wl.dtype)
            assert_close(f"{wl.name} dV[{b},{h}]", dV[b, h, rows], rV, wl.dtype)


def test_video_full_size_every_head_band_edges():
    _every_head_band_edges(WORKLOADS["video"], nrows=64, seed=101)


def test_train_full_size_fwd_bwd_sampled():
    _sampled(WORKLOADS["train"], nbh=24, nrows=40, seed=202, backward=True)


def test_long_full_size_every_head_band_edges():
    _every_head_band_edges(WORKLOADS["long"], nrows=48, seed=303)
