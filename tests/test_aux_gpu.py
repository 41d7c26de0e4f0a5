"""GPU tests of the library's auxiliary tools: the per-kernel timing print
(FIBATT_PROFILE=1) and the bounds-checked debug build (FIBATT_CHECKS=1).

The checks build runs a selection of the parity tests in a child process
(the binding loads one library per process): small and odd-sized cases on
every kernel family, the global first token, last-wave pieces and the
near-window forward, each against the oracle, and finally the device error
word, which a failed bounds check would have set.
"""
import os
import re
import subprocess
import sys

import pytest
import torch

from gpu_helpers import make_inputs, support_for, to_dev
from sparse_head_self_gb300 import api
from sparse_head_self_gb300.build import LIB_CHECKS
from sparse_head_self_gb300.inputs import WORKLOADS

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _profile_lines(err):
    out = {}
    for line in err.splitlines():
        m = re.match(r"libfibatt profile: (\w+) (.+) ([0-9.]+) us$", line)
        if m:
            out.setdefault(m.group(1), []).append((m.group(2), float(m.group(3))))
    return out


@pytest.mark.parametrize("name,B,kernels", [
    ("vitb", 2, {"fibatt_fwd": ["fwd_pipe_kernel"], "fibatt_bwd": ["bwd_pipe_kernel"]}),
    ("video", 1, {"fibatt_fwd": ["fwd_stream_kernel"],
                  "fibatt_bwd": ["rowdot_stream_kernel", "bwd_key_stream_kernel", "bwd_query_stream_kernel"]}),
])
def test_profile_prints_each_kernel(name, B, kernels, capfd, monkeypatch):
    monkeypatch.setenv("FIBATT_PROFILE", "1")
    monkeypatch.delenv("FIBATT_PATH", raising=False)
    wl = WORKLOADS[name].with_batch(B)
    q, k, v, do = make_inputs(wl, 3)
    sup = support_for(wl)
    qd, kd, vd, dod = to_dev(q, k, v, do)
    capfd.readouterr()
    O, L = api.fwd(sup, qd, kd, vd, wl.scale)
    api.bwd(sup, qd, kd, vd, O, L, dod, wl.scale)
    torch.cuda.synchronize()
    got = _profile_lines(capfd.readouterr().err)
    for call, names in kernels.items():
        assert [n.split("<")[0] for n, _ in got.get(call, [])] == names, (call, got)
        assert all(t > 0.0 for _, t in got[call]), got[call]


def test_profile_off_prints_nothing(capfd, monkeypatch):
    monkeypatch.delenv("FIBATT_PROFILE", raising=False)
    wl = WORKLOADS["tiny"]
    q, k, v, _ = make_inputs(wl, 4, with_grad=False)
    capfd.readouterr()
    api.fwd(support_for(wl), *to_dev(q, k, v), wl.scale)
    torch.cuda.synchronize()
    assert "libfibatt profile" not in capfd.readouterr().err


def test_checks_build_runs_the_parity_cases_clean():
    assert os.path.exists(LIB_CHECKS), "the checks build is made by __graft_entry__.build()"
    env = dict(os.environ, FIBATT_CHECKS="1")
    for k in ("FIBATT_PATH", "FIBATT_STREAM", "FIBATT_STREAM_WINDOW", "FIBATT_PROFILE"):
        env.pop(k, None)
    sel = ("tiny or edge_sizes or window_forward or vitb_shape_small or video_shape_two_heads or "
           "resident_bwd_last_wave_pieces or global_token_tiny or global_token_whole_heads_edge or "
           "global_token_whole_heads or no_device_error")
    r = subprocess.run([sys.executable, "-m", "pytest", "tests/test_parity_gpu.py", "-m", "gpu", "-x", "-q",
                        "-p", "no:cacheprovider", "-k", sel], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).splitlines()[-30:])
    assert r.returncode == 0, tail
    assert "libfibatt checks" not in r.stderr, tail
    assert re.search(r"\d+ passed", r.stdout), tail


def test_checks_build_is_the_library_loaded():
    # the child process of the test above loads the checks build
    code = ("import os; os.environ['FIBATT_CHECKS'] = '1'; "
            "from sparse_head_self_gb300 import _native; _native.lib(); print(_native.lib_path())")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == LIB_CHECKS
