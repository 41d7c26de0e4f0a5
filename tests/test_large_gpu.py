"""GPU parity at the size limits: tensors of more than 2^31 elements (so any
32-bit row or byte offset would wrap), on both the shared-memory kernels
(ViT-B heads) and the flat kernels (long windows), checked on sampled heads
at the far end of the tensors; and the largest head count with an offset
table near the entry limit.  The large cases allocate about 37 GB and skip
when the device has less free memory.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_close, oracle_heads
from sparse_head_self_gb300 import api
from sparse_head_self_gb300.inputs import WORKLOADS, Workload

pytestmark = pytest.mark.gpu

oracle.set_threads(oracle.max_threads())

ELEMS_2_31 = 2 ** 31


def _need_free(nbytes):
    free, _ = torch.cuda.mem_get_info()
    if free < nbytes:
        pytest.skip(f"needs {nbytes / 1e9:.0f} GB free on the device, {free / 1e9:.0f} GB free")


def _large_case(wl, heads_to_check, seed):
    n_elem = wl.B * wl.H * wl.N * wl.D
    assert n_elem > ELEMS_2_31
    _need_free(8.6 * n_elem * 2 + (4 << 30))
    g = torch.Generator(device="cuda").manual_seed(seed)
    shape = (wl.B, wl.H, wl.N, wl.D)
    q, k, v, do = (torch.randn(shape, device="cuda", dtype=torch.bfloat16, generator=g) for _ in range(4))
    sup = api.Support.wythoff(wl.H, wl.N, wl.w_min, wl.w_max, wl.diag)
    O, L = api.fwd(sup, q, k, v, wl.scale)
    dQ, dK, dV = api.bwd(sup, q, k, v, O, L, do, wl.scale)
    torch.cuda.synchronize()
    heads = oracle_heads(wl)
    for b, h in heads_to_check:
        hq, hk, hv, hdo = (x[b, h].float().cpu().numpy() for x in (q, k, v, do))
        Or, Lr = oracle.fwd_head(hq, hk, hv, heads[h], wl.scale)
        rQ, rK, rV = oracle.bwd_head(hq, hk, hv, hdo, heads[h], wl.scale)
        tag = f"{wl.name} b{b} h{h}"
        assert_close(f"{tag} O", O[b, h].float().cpu(), Or, "bf16")
        assert_close(f"{tag} LSE", L[b, h].cpu(), Lr, "bf16", lse=True)
        assert_close(f"{tag} dQ", dQ[b, h].float().cpu(), rQ, "bf16")
        assert_close(f"{tag} dK", dK[b, h].float().cpu(), rK, "bf16")
        assert_close(f"{tag} dV", dV[b, h].float().cpu(), rV, "bf16")
    del q, k, v, do, O, L, dQ, dK, dV
    torch.cuda.empty_cache()


def test_resident_kernels_beyond_2_31_elements():
    # ViT-B heads, B = 14200: 2.15e9 elements per tensor, 170,400 heads on
    # the persistent shared-memory kernels
    wl = WORKLOADS["vitb"].with_batch(14200)
    B, H = wl.B, wl.H
    _large_case(wl, [(B - 1, H - 1), (B - 1, 0), (B // 2, 5), (0, 0)], seed=71)


def test_flat_kernels_beyond_2_31_elements():
    # N = 4096, 16 heads with windows up to N (the flat kernels), B = 520:
    # 2.18e9 elements per tensor
    wl = Workload("wide", 520, 16, 4096, 64, "bf16", 64, 4096, True, True)
    B, H = wl.B, wl.H
    _large_case(wl, [(B - 1, H - 1), (B - 1, 3), (0, 0)], seed=72)


@pytest.mark.parametrize("path", ["generic", "resident", "flat"])
def test_sixty_four_heads_near_the_entry_limit(path, monkeypatch):
    # 64 heads (the maximum) of 7 distances each plus the diagonal: 960 of
    # the 1024 signed table entries; every output compared with the oracle
    # (N = 150 keeps a head's fp32 rows within one shared-memory stage)
    monkeypatch.setenv("FIBATT_PATH", path)
    N, H, B = 150, 64, 2
    rng = np.random.default_rng(5)
    dists = [sorted(rng.choice(np.arange(1, N), size=7, replace=False).tolist()) for _ in range(H)]
    sup = api.Support.from_distances(N, dists, True)
    assert sum(len(x) for x in sup.head_offsets()) == 960
    g = torch.Generator().manual_seed(6)
    q, k, v, do = (torch.randn(B, H, N, 64, generator=g) for _ in range(4))
    qd, kd, vd, dod = (x.cuda() for x in (q, k, v, do))
    O, L = api.fwd(sup, qd, kd, vd, 0.125)
    dQ, dK, dV = api.bwd(sup, qd, kd, vd, O, L, dod, 0.125)
    heads = [oracle.Head(d, N, True) for d in dists]
    Or, Lr = oracle.fwd(q, k, v, heads, 0.125)
    rQ, rK, rV = oracle.bwd(q, k, v, do, heads, 0.125)
    for name, got, ref in (("O", O, Or), ("dQ", dQ, rQ), ("dK", dK, rK), ("dV", dV, rV)):
        assert_close(f"64 heads {path} {name}", got.cpu(), ref, "f32")
    assert_close(f"64 heads {path} LSE", L.cpu(), Lr, "f32", lse=True)
