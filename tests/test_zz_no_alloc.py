"""The allocation-free route build (estream_route_build_noalloc).

It serves callers that cannot give the library device scratch memory (for
example a serving process that reserved all device memory up front and
allows no cudaMalloc on its request path). Its scratch is a static device
array shared by every call, so these tests check that two calls in a row --
with different sizes, the second one smaller -- each give exactly what the
workspace-taking estream_route_build gives, and that oversized requests are
refused. This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch


def _lib():
    from routed_expert_ffn_topk_gb300 import build as b
    b.build()
    from routed_expert_ffn_topk_gb300 import estream as es
    return es


def test_noalloc_rejects_sizes_beyond_its_scratch():
    es = _lib()
    L = es.lib()
    # 1 MiB of scratch: 4096 slots x 64 chunks of routes is far beyond it
    T, E, k, P = 65536, 1024, 1, 4096
    assert es.route_workspace_bytes(T, E, k, P) > (1 << 20)
    st = L.estream_route_build_noalloc(ctypes.c_void_p(16), T, E, k, 0, ctypes.c_void_p(16), P,
                                       ctypes.c_void_p(16), ctypes.c_void_p(16), ctypes.c_void_p(16),
                                       ctypes.c_void_p(16), ctypes.c_void_p(16), None)
    assert st == es.ERR_CAPACITY
    st = L.estream_route_build_noalloc(None, 4, 8, 9, 0, None, 8, None, None, None, None, None, None)
    assert st == es.ERR_INVALID_ARG


@pytest.mark.gpu
def test_noalloc_matches_workspace_route_build_twice():
    es = _lib()
    dev = torch.device("cuda", 0)
    cases = [(2048, 64, 8, True, 24), (300, 60, 4, False, 60)]   # second call smaller
    for T, E, k, renorm, P in cases:
        g = torch.Generator().manual_seed(T + E)
        lg = torch.randn(T, E, generator=g).to(dev)
        phi = None
        if P != E:
            perm = torch.randperm(E, generator=g)
            phi_h = torch.full((E,), -1, dtype=torch.int32)
            phi_h[perm[:P]] = torch.arange(P, dtype=torch.int32)
            phi = phi_h.to(dev)
        ref = es.route_build(lg, k, renorm, phi, P)
        got = es.route_build_noalloc(lg, k, renorm, phi, P)
        torch.cuda.synchronize()
        R = T * k
        for name in ("topk_ids", "rec_tok", "rec_route"):
            assert torch.equal(got[name][:R], ref[name][:R]), name
        assert torch.equal(got["offsets"], ref["offsets"])
        assert torch.equal(got["alpha"][:R].view(torch.int32), ref["alpha"][:R].view(torch.int32))
