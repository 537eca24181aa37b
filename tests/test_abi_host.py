"""C ABI and host-side logic of libestream, without a GPU.

Checks that the library loads and exports every function include/estream.h
declares, that argument errors come back as status codes before anything
touches CUDA, and that the offline expert packer lays groups out as the
pager expects (with an exact fp16 conversion of the down plane).
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "estream.h")


@pytest.fixture(scope="module")
def es():
    build_mod.build()
    from routed_expert_ffn_topk_gb300 import estream
    estream.lib()
    return estream


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(estream_[a-z0-9_]+)\s*\(", text)))


def test_header_symbols_exported(es):
    names = declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(es.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), f"{n} declared in estream.h but not exported"
        assert n in es.SIGNATURES, f"{n} has no Python binding"


def test_status_strings(es):
    assert es.status_string(es.OK) == "ok"
    assert "capacity" in es.status_string(es.ERR_CAPACITY)
    assert es.version() >= 10000


def test_route_build_argument_errors(es):
    L = es.lib()
    ws = ctypes.create_string_buffer(4096)
    # k > E, k < 1, E > 1024, P != E without phi, P > 4096
    for (T, E, k, P) in [(4, 8, 9, 8), (4, 8, 0, 8), (4, 2000, 2, 2000), (4, 8, 2, 6), (4, 8, 2, 5000)]:
        st = L.estream_route_build(None, T, E, k, 0, None, P, None, None, None, None, None,
                                   ctypes.addressof(ws), 4096, None)
        assert st == es.ERR_INVALID_ARG, (T, E, k, P, st)
    # null outputs with T > 0
    st = L.estream_route_build(None, 4, 8, 2, 0, None, 8, None, None, ctypes.addressof(ws),
                               None, None, ctypes.addressof(ws), 4096, None)
    assert st == es.ERR_INVALID_ARG
    assert es.route_workspace_bytes(4096, 64, 8, 64) > es.route_workspace_bytes(64, 64, 8, 64) > 0
    assert es.route_workspace_bytes(4, 8, 2, -1) == 0


def test_layer_calls_need_context(es):
    L = es.lib()
    assert L.estream_moe_layer_prefill(None, 0, None, None, 1, 1, 0, None, None) == es.ERR_NOT_BOUND
    assert L.estream_arena_preload(None, 0, None) == es.ERR_NOT_BOUND
    assert L.estream_get_device_error(None) == es.ERR_NOT_BOUND
    assert L.estream_moe_layer_prefill_residual(None, 0, None, None, 1, 1, 0, None, None,
                                                None) == es.ERR_NOT_BOUND
    assert L.estream_inject_route_timeout(None) == es.ERR_NOT_BOUND
    assert L.estream_inject_expert_timeout(None) == es.ERR_NOT_BOUND
    assert L.estream_inject_pager_fault(None, 0, 0) == es.ERR_NOT_BOUND
    out = ctypes.c_void_p()
    assert L.estream_bind_arena(ctypes.byref(out), None) == es.ERR_INVALID_ARG
    L.estream_unbind(None)  # no-op


def _desc(es, **kw):
    base = dict(L=1, E=8, H=256, F=128, G=4, B=2, wdtype=es.BF16)
    base.update(kw)
    d = es.ArenaDesc()
    for k, v in base.items():
        setattr(d, k, v)
    d.Q, d.T_max, d.k_max = 1, 16, 2
    return d


def test_bind_rejects_bad_shapes_before_cuda(es):
    L = es.lib()
    out = ctypes.c_void_p()
    for kw in (dict(H=200), dict(F=100), dict(E=0), dict(G=0), dict(B=0), dict(wdtype=7)):
        d = _desc(es, **kw)
        st = L.estream_bind_arena(ctypes.byref(out), ctypes.byref(d))
        assert st in (es.ERR_INVALID_ARG, es.ERR_UNSUPPORTED), (kw, st)
    d = _desc(es)  # valid shape but no arena / pools
    assert L.estream_bind_arena(ctypes.byref(out), ctypes.byref(d)) == es.ERR_INVALID_ARG


def test_sizes(es):
    assert es.arena_bytes(64, 2048, 1024, 8, 2, es.BF16) == 16 * 3 * 2048 * 1024 * 2
    assert es.pool_bytes(60, 2048, 1408, es.BF16) == 60 * 3 * 2048 * 1408 * 2 + 240
    assert es.shared_bytes(2, 2048, 1408, es.BF16) == 2 * 3 * 2048 * 1408 * 2 + 16


def untile(flat, rows, cols, tile_rows):
    """Inverse of the tile-major plane layout [rows/tr][cols/64][tr][64]."""
    t = flat.reshape(rows // tile_rows, cols // 64, tile_rows, 64)
    return t.transpose(0, 2, 1, 3).reshape(rows, cols)


def _bf16_bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("G", [1, 3, 4, 8])
def test_pack_experts_layout(es, G):
    """Group q holds the experts at storage positions [qG, qG+G) in order,
    as [gate][up][down], each plane tile-major (128-row tiles for gate/up,
    256-row tiles for down, 64 columns each); the down plane is
    fp16(W_d * 2^s) with the scale 2^-s stored after the groups, and converts
    back exactly."""
    E, H, F = 7, 256, 128
    g = torch.Generator().manual_seed(3)
    Wg = (torch.randn(E, F, H, generator=g) * 0.02).bfloat16()
    Wu = (torch.randn(E, F, H, generator=g) * 0.02).bfloat16()
    Wd = (torch.randn(E, H, F, generator=g) * 0.02).bfloat16()
    Wd[2] *= 1000.0  # a different scale per expert
    perm = torch.randperm(E, generator=g).to(torch.int32)
    d, keep = es.make_desc(1, E, H, F, G, 1, es.BF16, None, [None], perm=perm)
    pool = torch.zeros(es.pool_bytes(E, H, F, es.BF16), dtype=torch.uint8)
    es.pack_experts(d, 0, Wg, Wu, Wd, pool)
    raw = pool.numpy()
    S = H * F * 2
    W = 3 * S
    scales = raw[E * W:E * W + 4 * E].view(np.float32)
    for e in range(E):
        pos = int(perm[e])
        q, r = divmod(pos, G)
        n_q = min(G, E - q * G)
        base = q * G * W
        gate = untile(raw[base + r * S: base + (r + 1) * S].view(np.uint16), F, H, 128)
        up = untile(raw[base + n_q * S + r * S: base + n_q * S + (r + 1) * S].view(np.uint16), F, H, 128)
        down = untile(raw[base + 2 * n_q * S + r * S: base + 2 * n_q * S + (r + 1) * S].view(np.float16),
                      H, F, 256)
        np.testing.assert_array_equal(gate, _bf16_bits(Wg[e]))
        np.testing.assert_array_equal(up, _bf16_bits(Wu[e]))
        sc = float(scales[pos])
        assert sc > 0 and np.log2(sc) == int(np.log2(sc))      # a power of two
        back = down.astype(np.float64) * sc
        np.testing.assert_array_equal(back, Wd[e].double().numpy())
        assert 2.0 ** 14 <= np.abs(down.astype(np.float64)).max() < 2.0 ** 15


def test_pack_rejects_bad_perm(es):
    E, H, F = 4, 256, 128
    z = torch.zeros(E, F, H, dtype=torch.bfloat16)
    zd = torch.zeros(E, H, F, dtype=torch.bfloat16)
    d, keep = es.make_desc(1, E, H, F, 2, 1, es.BF16, None, [None], perm=[0, 1, 1, 3])
    pool = torch.zeros(es.pool_bytes(E, H, F, es.BF16), dtype=torch.uint8)
    with pytest.raises(es.EStreamError):
        es.pack_experts(d, 0, z, z, zd, pool)


def test_layer_call_argument_checks(es):
    """The binding rejects tensors whose shapes or types do not fit the layer
    call before any pointer reaches the library."""
    import pytest
    import torch
    T, H, E = 8, 256, 4
    X = torch.zeros(T, H, dtype=torch.bfloat16)
    lg = torch.zeros(T, E, dtype=torch.float32)
    Y = torch.zeros(T, H, dtype=torch.float32)
    bad = [
        (X, lg, torch.zeros(T, H + 1), None),               # Y shape
        (X, torch.zeros(T + 1, E), Y, None),                # logits rows
        (X, lg.double(), Y, None),                          # logits type
        (X, lg, Y.half(), None),                            # Y type
        (X.int(), lg, Y, None),                             # X type
        (X, lg, Y, torch.zeros(T, H, dtype=torch.float32)), # residual type
        (X, lg, Y, torch.zeros(T, H - 1, dtype=torch.bfloat16)),
        (X, lg, Y, None),                                   # not on a CUDA device
    ]
    for x, l, y, a in bad:
        with pytest.raises(ValueError):
            if a is None:
                es.moe_layer_prefill(None, 0, x, l, 2, False, y)
            else:
                es.moe_layer_prefill_residual(None, 0, x, l, 2, False, a, y)


def test_route_and_router_argument_checks(es):
    """The route build and router wrappers reject tensors that do not fit
    before any pointer reaches the library."""
    import pytest
    import torch
    with pytest.raises(ValueError):
        es.route_build(torch.zeros(4, 8), 2, False)                       # not on a CUDA device
    with pytest.raises(ValueError):
        es.route_build(torch.zeros(4, 8, dtype=torch.float64), 2, False)  # not fp32
    with pytest.raises(ValueError):
        es.route_build_noalloc(torch.zeros(8), 2, False)                  # not 2-d
    X = torch.zeros(4, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        es.router_logits(X, torch.zeros(8, 64, dtype=torch.bfloat16))     # H differs
    with pytest.raises(ValueError):
        es.router_logits(X, torch.zeros(8, 128))                          # W_r not bf16
    with pytest.raises(ValueError):
        es.router_logits(X, torch.zeros(8, 128, dtype=torch.bfloat16))    # not on a CUDA device
