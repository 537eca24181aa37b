"""Router logits upstream of the top-k (l = X W_r^T, bf16 in, fp32 out) on
the tensor cores against the fp64 oracle, and the top-k taken from them."""
import numpy as np
import pytest
import torch

import oracle
from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


def _bound(X, W_r):
    """|GPU - exact| <= (H/16 + 64) * 2^-24 * sum_h |x_h w_h|: the products of
    two bf16 values are exact in fp32; each logit is a sum of H/16 fp32
    accumulation steps of 16-term tensor-core dot products plus at most H/64
    split partials added in fp32, each step adding at most one rounding of
    2^-24 relative to the running magnitude, itself at most sum |x w|
    (at most 8 partial sums are added, fewer than H/64 + 64)."""
    H = X.shape[1]
    a = np.abs(X.float().numpy()).astype(np.float64) @ np.abs(W_r.float().numpy()).astype(np.float64).T
    return (H / 16 + 64) * 2.0 ** -24 * a


def _gpu_logits(X, W_r):
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = _gpu.device()
    ws = torch.empty(max(es.router_workspace_bytes(X.shape[0], X.shape[1], W_r.shape[0]), 256),
                     dtype=torch.uint8, device=dev)
    out = es.router_logits(X.to(dev), W_r.to(dev), workspace=ws)
    assert es.workspace_error(ws) == es.OK
    return out.cpu()


@pytest.mark.parametrize("T,H,E", [(1, 64, 8), (129, 128, 60), (1024, 2048, 64), (2048, 2048, 64),
                                   (4096, 2048, 60), (4096, 4096, 8), (300, 256, 300),
                                   (257, 512, 1024)])
def test_router_logits_vs_oracle(T, H, E):
    X, W_r = W.make_router(T, H, E, seed=1700 + E)
    got = _gpu_logits(X, W_r).numpy().astype(np.float64)
    ref = oracle.router_logits(X, W_r)
    err = np.abs(got - ref)
    bound = _bound(X, W_r)
    assert np.all(err <= bound), f"max excess {(err - bound).max():.3e}"


def test_router_logits_deterministic():
    X, W_r = W.make_router(1024, 2048, 64, seed=5)
    a = _gpu_logits(X, W_r)
    b = _gpu_logits(X, W_r)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


@pytest.mark.parametrize("T,H,E,k,renorm", [(1024, 2048, 64, 8, False), (4096, 4096, 8, 2, True)])
def test_topk_from_router_logits(T, H, E, k, renorm):
    """The top-k taken on the GPU from its own logits equals the oracle's
    top-k of the same logits bit for bit, and is a valid top-k of the exact
    logits up to the accumulation bound (near-ties may order either way)."""
    from routed_expert_ffn_topk_gb300 import estream as es
    X, W_r = W.make_router(T, H, E, seed=99)
    lg = _gpu_logits(X, W_r)
    out = es.route_build(lg.to(_gpu.device()), k, renorm)
    ids = out["topk_ids"].cpu().numpy().reshape(T, k)
    alpha = out["alpha"].cpu().numpy().reshape(T, k)
    ids_o, alpha_o = oracle.route_topk(lg.numpy(), k, renorm)
    np.testing.assert_array_equal(ids, ids_o)
    np.testing.assert_array_equal(alpha.view(np.uint32), alpha_o.view(np.uint32))
    exact = oracle.router_logits(X, W_r)
    bound = _bound(X, W_r)
    # GPU logit g and exact logit x differ by at most b, so a selected s and
    # an unselected u must satisfy x_s + b_s >= x_u - b_u
    for t in range(T):
        sel = np.zeros(E, bool)
        sel[ids[t]] = True
        if sel.all():
            continue
        assert (exact[t, sel] + bound[t, sel]).min() >= (exact[t, ~sel] - bound[t, ~sel]).max(), t


def test_router_argument_errors():
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = _gpu.device()
    X = torch.zeros(4, 96, dtype=torch.bfloat16, device=dev)
    Wr = torch.zeros(8, 96, dtype=torch.bfloat16, device=dev)
    with pytest.raises(es.EStreamError) as ei:
        es.router_logits(X, Wr)                      # H not a multiple of 64
    assert ei.value.status == es.ERR_INVALID_ARG
    X = torch.zeros(1024, 2048, dtype=torch.bfloat16, device=dev)
    Wr = torch.zeros(64, 2048, dtype=torch.bfloat16, device=dev)
    small = torch.empty(128, dtype=torch.uint8, device=dev)
    assert es.router_workspace_bytes(1024, 2048, 64) == 256   # the error word only
    with pytest.raises(es.EStreamError) as ei:
        es.router_logits(X, Wr, workspace=small)
    assert ei.value.status == es.ERR_CAPACITY


def test_layer_from_router():
    """X -> router logits -> top-k -> fused experts -> Y, checked against the
    oracle layer fed the GPU's logits (the logits themselves are checked
    above)."""
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    from tests.test_gpu_layer import small_workload
    wl = small_workload("c3")
    cfg = wl.cfg
    _, W_r = W.make_router(1, cfg.H, cfg.E, seed=31)
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode="paged")
    try:
        Y = torch.zeros(cfg.T, cfg.H, dtype=torch.float32, device=dev)
        lg = st.prefill_from_router(0, wl.X.to(dev), W_r.to(dev), Y)
        torch.cuda.synchronize()
        lg = lg.cpu().clone()
        y = Y.cpu().numpy()
    finally:
        st.close()
    np.testing.assert_allclose(lg.numpy(), oracle.router_logits(wl.X, W_r), rtol=0,
                               atol=float(_bound(wl.X, W_r).max()))
    wl2 = W.Workload(cfg, [lg], wl.X, wl.layers)
    ref = _gpu.oracle_layer(wl2, 0, wl.X)
    _gpu.assert_y_close(y, ref, "layer from router")
