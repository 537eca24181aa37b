"""Routing from the layer input in one launch (estream_route_build_from_x,
estream_moe_layer_prefill_from_x): router logits X W_r^T on the tensor cores,
reduced over a thread-block cluster, ranked in shared memory and turned into
the route map by the same grid-wide construction as estream_route_build.

Checked against the oracle: the logits within the accumulation bound of
the fp64 router, and the top-k, alpha and route map bit for bit against the
oracle's top-k and Algorithm 1 run on the GPU's own logits (the logits are
what the GPU ranks; near-ties of the exact logits may order either way, and
the router tests check that the ranking is a valid top-k of the exact ones).
"""
import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu
from tests.test_gpu_router import _bound

pytestmark = pytest.mark.gpu


def _from_x(X, W_r, k, renorm, phi=None, P=None):
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = _gpu.device()
    ph = None if phi is None else torch.as_tensor(phi, dtype=torch.int32).to(dev)
    out = es.route_build_from_x(X.to(dev), W_r.to(dev), k, renorm, ph, P)
    assert es.workspace_error(out["workspace"]) == es.OK
    T = X.shape[0]
    R = T * k
    return {n: out[n].cpu() if n in ("logits", "offsets") else out[n].cpu()[:R]
            for n in ("logits", "topk_ids", "alpha", "offsets", "rec_tok", "rec_route")}


def _check(X, W_r, k, renorm, phi=None, P=None):
    T, E = X.shape[0], W_r.shape[0]
    P = E if P is None else P
    got = _from_x(X, W_r, k, renorm, phi, P)
    lg = got["logits"].numpy()
    err = np.abs(lg.astype(np.float64) - oracle.router_logits(X, W_r))
    assert np.all(err <= _bound(X, W_r)), "logits beyond the accumulation bound"
    ids, alpha = oracle.route_topk(lg, k, renorm)
    offs, rt, rr = oracle.route_csr(ids, E, P, phi)
    np.testing.assert_array_equal(got["topk_ids"].numpy(), ids.ravel())
    np.testing.assert_array_equal(got["alpha"].numpy().view(np.uint32), alpha.ravel().view(np.uint32))
    np.testing.assert_array_equal(got["offsets"].numpy(), offs)
    np.testing.assert_array_equal(got["rec_tok"].numpy(), rt)
    np.testing.assert_array_equal(got["rec_route"].numpy(), rr)
    return got


@pytest.mark.parametrize("T,H,E,k,renorm,fused", [
    (1024, 2048, 64, 8, False, True),    # OLMoE-shaped
    (2048, 2048, 64, 6, True, True),     # DeepSeek-V2-Lite-shaped
    (4096, 2048, 60, 4, False, True),    # Qwen-MoE-shaped
    (4096, 4096, 8, 2, True, True),      # Mixtral-shaped
    (129, 128, 60, 4, False, True),      # ragged last tile, one k-split
    (1, 64, 8, 2, False, True),          # one token
    (300, 256, 128, 16, True, True),     # largest E of the fused form
    (257, 512, 300, 6, False, False),    # E > 128: router + route build
])
def test_route_from_x_vs_oracle(T, H, E, k, renorm, fused):
    from routed_expert_ffn_topk_gb300 import estream as es
    assert es.route_build_from_x_fused(T, H, E) == fused
    X, W_r = W.make_router(T, H, E, seed=2100 + E + T)
    _check(X, W_r, k, renorm)


def test_route_from_x_partial_placement():
    """Phi a random partial injection into P < E slots: unresolved routes in
    the trailing bucket, as in Algorithm 1's reading."""
    T, H, E, k, P = 700, 512, 64, 6, 24
    X, W_r = W.make_router(T, H, E, seed=77)
    g = torch.Generator().manual_seed(4)
    perm = torch.randperm(E, generator=g)
    phi = torch.full((E,), -1, dtype=torch.int32)
    phi[perm[:P]] = torch.arange(P, dtype=torch.int32)
    _check(X, W_r, k, False, phi=phi.numpy(), P=P)


def test_route_from_x_matches_two_launches_on_its_logits():
    """The route map of the single launch equals estream_route_build run on
    the logits the single launch wrote, bit for bit, on consecutive calls
    with different inputs and a poisoned workspace in between."""
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = _gpu.device()
    T, H, E, k = 2048, 2048, 64, 6
    ws = torch.empty(es.route_workspace_bytes(T, E, k, E), dtype=torch.uint8, device=dev)
    for seed in (5, 6):
        X, W_r = W.make_router(T, H, E, seed=seed)
        ws.fill_(0xFF)
        got = es.route_build_from_x(X.to(dev), W_r.to(dev), k, True, workspace=ws)
        assert es.workspace_error(ws) == es.OK
        ref = es.route_build(got["logits"].clone(), k, True)
        torch.cuda.synchronize()
        for n in ("topk_ids", "alpha", "offsets", "rec_tok", "rec_route"):
            assert torch.equal(got[n].view(torch.int32), ref[n].view(torch.int32)), n


@pytest.mark.parametrize("mode,residual", [("resident", True), ("paged", False), ("resident", False)])
def test_layer_prefill_from_x(mode, residual):
    """X and W_r -> one routing launch -> fused experts -> Y, against the
    oracle layer fed the GPU's logits; the logits the call returns are the
    ones estream_route_build_from_x writes for the same X and W_r."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    from tests.test_gpu_layer import small_workload
    wl = small_workload("c3")
    cfg = wl.cfg
    _, W_r = W.make_router(1, cfg.H, cfg.E, seed=33)
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode=mode)
    try:
        X = wl.X.to(dev)
        Y = torch.full((cfg.T, cfg.H), float("nan") if residual else 0.0, device=dev)
        lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
        st.poison()
        st.prefill_from_x(0, X, W_r.to(dev), Y, residual=X if residual else None, logits_out=lg)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        y = Y.cpu().numpy()
        lg_cpu = lg.cpu()
    finally:
        st.close()
    same = es.route_build_from_x(X, W_r.to(dev), cfg.k, cfg.renorm)["logits"].cpu()
    assert torch.equal(lg_cpu.view(torch.int32), same.view(torch.int32))
    wl2 = W.Workload(cfg, [lg_cpu], wl.X, wl.layers)
    A = wl.X.double().numpy() if residual else None
    ref = _gpu.oracle_layer(wl2, 0, wl.X, residual=A)
    if residual:
        y, ref = y - A, ref - A
    _gpu.assert_y_close(y, ref, f"layer from X ({mode}, residual={residual})")


def test_layer_prefill_from_x_full_size():
    """The OLMoE-shaped layer at full size, resident, routed from X in one
    launch, on rows covering every m-block of its route map."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.CONFIGS["c2"]
    wl = W.make_workload(cfg)
    _, W_r = W.make_router(1, cfg.H, cfg.E, seed=35)
    dev = _gpu.device()
    assert es.route_build_from_x_fused(cfg.T, cfg.H, cfg.E)
    st = BoundLayerStack(wl, mode="resident")
    try:
        X = wl.X.to(dev)
        Y = torch.empty(cfg.T, cfg.H, device=dev)
        lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
        st.poison()
        st.prefill_from_x(0, X, W_r.to(dev), Y, residual=X, logits_out=lg)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        y = Y.cpu().numpy()
        lg_cpu = lg.cpu()
    finally:
        st.close()
    rows = _gpu.rows_covering_mblocks(lg_cpu.numpy(), cfg.k)
    wl2 = W.Workload(cfg, [lg_cpu], wl.X, wl.layers)
    A = wl.X.double().numpy()
    ref = _gpu.oracle_layer(wl2, 0, wl.X, rows=rows, residual=A)
    _gpu.assert_y_close(y[rows] - A[rows], ref - A[rows], f"c2 from X, {len(rows)} rows")


def test_layer_from_x_route_timeout_then_normal():
    """The single routing launch's bounded grid barrier: one CTA withholds its
    arrival (estream_inject_route_timeout), the others' 1 s wait runs out,
    the call leaves an empty route map (Y = the residual rows), reports
    ESTREAM_ERR_TIMEOUT, and the next call is normal. No GPU fault."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    from tests.test_gpu_layer import small_workload
    wl = small_workload("c2")
    cfg = wl.cfg
    _, W_r = W.make_router(1, cfg.H, cfg.E, seed=36)
    dev = _gpu.device()
    assert es.route_build_from_x_fused(cfg.T, cfg.H, cfg.E)
    st = BoundLayerStack(wl, mode="resident")
    try:
        X = wl.X.to(dev)
        Y = torch.empty(cfg.T, cfg.H, device=dev)
        es.inject_route_timeout(st.ctx)
        st.prefill_from_x(0, X, W_r.to(dev), Y, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.ERR_TIMEOUT
        assert torch.equal(Y, X.float())
        lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
        st.prefill_from_x(0, X, W_r.to(dev), Y, residual=X, logits_out=lg)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        y = Y.cpu().numpy()
        lg_cpu = lg.cpu()
    finally:
        st.close()
    wl2 = W.Workload(cfg, [lg_cpu], wl.X, wl.layers)
    A = wl.X.double().numpy()
    ref = _gpu.oracle_layer(wl2, 0, wl.X, residual=A)
    _gpu.assert_y_close(y - A, ref - A, "c2 from X after a route timeout")


def test_layer_from_x_residual_at_4096():
    """A layer call routed from X at T = 4096 with a residual: the rows go to
    the first expert launch (more than the routing launch covers beside its
    router tile). Y - A against the oracle fed the GPU's logits, on every row,
    with the workspace poisoned before the call."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.scaled(W.CONFIGS["c5"], T=4096, H=256, E=8, k=2, F=256, key_suffix="-fromx4096")
    wl = W.make_workload(cfg, seed=4097)
    _, W_r = W.make_router(1, cfg.H, cfg.E, seed=37)
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode="resident")
    try:
        X = wl.X.to(dev)
        A = torch.randn(X.shape, generator=torch.Generator().manual_seed(6), dtype=torch.float32)
        A = A.to(X.dtype).to(dev)
        Y = torch.full((cfg.T, cfg.H), float("nan"), device=dev)
        lg = torch.empty(cfg.T, cfg.E, dtype=torch.float32, device=dev)
        st.poison()
        st.prefill_from_x(0, X, W_r.to(dev), Y, residual=A, logits_out=lg)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        y = Y.cpu().numpy()
        lg_cpu = lg.cpu()
    finally:
        st.close()
    wl2 = W.Workload(cfg, [lg_cpu], wl.X, wl.layers)
    Ac = A.cpu().double().numpy()
    ref = _gpu.oracle_layer(wl2, 0, wl.X)
    _gpu.assert_y_close(y - Ac, ref, "from X, T = 4096, residual in the expert launch")
