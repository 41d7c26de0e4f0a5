"""fibatt_bwd_noalloc against fibatt_bwd, through the C ABI.

fibatt_bwd_noalloc exists for callers that cannot allocate device memory (no
allocator at hand, or not allowed to use it at that point): it takes no
workspace and keeps its per-row scratch in a fixed array inside the library.
Its results must match the ordinary backward entry point within the tests'
tolerances, on consecutive calls (the array keeps the previous call's
contents, which the next call must not depend on).

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import TOL, make_inputs, support_for, to_dev
from sparse_head_self_gb300 import _native, api
from sparse_head_self_gb300.inputs import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


def _noalloc(sup, wl, q, k, v, o, lse, do, dq, dk, dv):
    L = _native.lib()
    dt = _native.F32 if wl.dtype == "f32" else _native.BF16
    st = L.fibatt_bwd_noalloc(sup.handle, wl.B, wl.D, dt, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                              o.data_ptr(), lse.data_ptr(), do.data_ptr(), wl.scale, dq.data_ptr(),
                              dk.data_ptr(), dv.data_ptr(), torch.cuda.current_stream().cuda_stream)
    _native.check(st)


def _close(name, got, ref, dtype):
    d = (got.double() - ref.double()).abs().cpu().numpy()
    t = TOL[dtype]
    assert d.max() <= t["max_abs"], f"{name}: max-abs {d.max():.3e}"
    if dtype == "bf16":
        assert d.mean() <= t["mean_abs"], f"{name}: mean-abs {d.mean():.3e}"


@pytest.mark.parametrize("wl", [WORKLOADS["tiny"],
                                Workload(**{**WORKLOADS["vitb"].__dict__, "B": 3}),
                                Workload(**{**WORKLOADS["video"].__dict__, "B": 1})],
                         ids=["tiny_f32", "vitb_bf16", "video_bf16"])
def test_noalloc_matches_bwd_on_two_calls(wl):
    q, k, v, do = make_inputs(wl, 41)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    o, lse = api.fwd(sup, qd, kd, vd, wl.scale)
    ref = api.bwd(sup, qd, kd, vd, o, lse, dod, wl.scale)
    outs = []
    for call in range(2):
        dq, dk, dv = (torch.full_like(qd, float("nan")) for _ in range(3))
        _noalloc(sup, wl, qd, kd, vd, o, lse, dod, dq, dk, dv)
        torch.cuda.synchronize()
        for name, g, r in zip(("dQ", "dK", "dV"), (dq, dk, dv), ref):
            _close(f"call {call} {name}", g, r, wl.dtype)
        outs.append((dq, dk, dv))
    for a, b in zip(*outs):
        assert torch.equal(a, b)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # N * H * B above the fixed scratch: refused before anything is launched
    N, H = 4096, 1
    B = (1 << 20) // (N * H) + 1
    sup = api.Support.build(N, [1], [2], [100], True)
    t = torch.empty(64, dtype=torch.bfloat16, device="cuda")   # never touched: the size check fails first
    L = _native.lib()
    p = t.data_ptr()
    st = L.fibatt_bwd_noalloc(sup.handle, B, 64, _native.BF16, p, p, p, p, p, p, 0.125, p, p, p, None)
    assert st == 1
    assert "exceed" in L.fibatt_last_error().decode()
