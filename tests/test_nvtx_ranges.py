"""NVTX ranges of the runtime (domain "estream"), for timeline tools.

The ranges are recorded by an NVTX injection library built from
tests/nvtx/nvtx_record.c, which NVTX loads in a child process through the
NVTX_INJECTION64_PATH environment variable. Each range's name is a string
registered once, and its payload holds the layer (bank fills: layer * 65536 +
group).

Without a GPU: the standalone calls open their range before they validate
their arguments, so an invalid route build and a preload without a context
record balanced ranges. On a GPU: a paged, deterministic layer call with
shared experts records, nested in its "layer" range, the route build, one
bank fill per expert group, the routed and shared expert launches and the
combine; a layer call from the layer input records "route from X" inside its
route build.
"""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "nvtx", "nvtx_record.c")


def _cuda_include():
    for base in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if base and os.path.isfile(os.path.join(base, "include", "nvtx3", "nvToolsExt.h")):
            return os.path.join(base, "include")
    return None


@pytest.fixture(scope="module")
def recorder(tmp_path_factory):
    inc = _cuda_include()
    if shutil.which("gcc") is None or inc is None:
        pytest.skip("gcc or the NVTX3 headers are not available")
    out = str(tmp_path_factory.mktemp("nvtx") / "libnvtx_record.so")
    subprocess.run(["gcc", "-shared", "-fPIC", "-O2", "-I" + inc, "-o", out, SRC, "-lpthread"],
                   check=True, capture_output=True)
    from routed_expert_ffn_topk_gb300 import build as build_mod
    build_mod.build()
    return out


def _record(recorder, tmp_path, code, timeout=600):
    path = str(tmp_path / "ranges.txt")
    env = dict(os.environ, NVTX_INJECTION64_PATH=recorder, NVTX_RECORD_PATH=path)
    env["PYTHONPATH"] = ROOT + os.pathsep + env.get("PYTHONPATH", "")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, timeout=timeout,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    return open(path).read().splitlines() if os.path.exists(path) else []


def _tree(lines):
    """(name, payload, parent name) of every estream range, checking that
    pushes and pops balance."""
    stack, ranges = [], []
    for ln in lines:
        parts = ln.split(" ")
        if parts[0] == "push" and parts[1] == "estream":
            name, payload = " ".join(parts[2:-1]), int(parts[-1])
            ranges.append((name, payload, stack[-1][0] if stack else None))
            stack.append((name, payload))
        elif parts[0] == "pop" and parts[1] == "estream":
            assert stack, "pop without a push"
            stack.pop()
    assert not stack, f"ranges left open: {stack}"
    return ranges


def test_ranges_of_standalone_calls(recorder, tmp_path):
    code = """
import ctypes
from routed_expert_ffn_topk_gb300 import estream as es
L = es.lib()
ws = ctypes.create_string_buffer(4096)
st = L.estream_route_build(None, 4, 8, 9, 0, None, 8, None, None, None, None, None,
                           ctypes.addressof(ws), 4096, None)
assert st == es.ERR_INVALID_ARG, st
assert L.estream_arena_preload(None, 2, None) == es.ERR_NOT_BOUND
"""
    lines = _record(recorder, tmp_path, code)
    assert "domain estream" in lines
    assert _tree(lines) == [("route build", -1, None), ("preload", 2, None)]


@pytest.mark.gpu
def test_ranges_of_a_layer_call(recorder, tmp_path):
    code = """
import torch
from routed_expert_ffn_topk_gb300 import estream as es, workloads as W
from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
cfg = W.scaled(W.CONFIGS["c3"], T=320, H=512, E=12, k=3, F=256, F_shared=384)
wl = W.make_workload(cfg)
st = BoundLayerStack(wl, mode="paged", deterministic=True, G=4, B=2)
X, lg = wl.X.cuda(), wl.logits[0].cuda()
Y = torch.zeros(cfg.T, cfg.H, device="cuda")
st.prefill(0, X, lg, Y)
_, W_r = W.make_router(1, cfg.H, cfg.E, seed=33)
st.prefill_from_x(0, X, W_r.cuda(), Y)
torch.cuda.synchronize()
assert es.get_device_error(st.ctx) == es.OK
st.close()
"""
    ranges = _tree(_record(recorder, tmp_path, code))
    layers = [r for r in ranges if r[0] == "layer"]
    assert [(p, parent) for _, p, parent in layers] == [(0, None), (0, None)]
    inner = [(n, p) for n, p, parent in ranges if parent == "layer"]
    assert inner.count(("route build", 0)) == 2
    # 12 experts in groups of 4 through 2 banks: one fill per group, per call
    fills = sorted(p for n, p in inner if n == "bank fill")
    assert fills == [0, 0, 1, 1, 2, 2], fills
    assert inner.count(("routed experts", 0)) >= 2
    assert inner.count(("shared experts", 0)) == 2
    assert inner.count(("combine", 0)) == 2
    assert [(n, p, parent) for n, p, parent in ranges if n == "route from X"] == \
        [("route from X", 0, "route build")]
