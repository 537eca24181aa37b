"""One MoE layer's prefill through the C ABI against the oracle.

Small shapes of every model family are compared element by element (all of
Y); the full-size layer shapes are compared on token rows that the oracle
evaluates one by one, chosen so that every (expert, 128-record block) of the
route map holds a checked record.
"""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu

# (family, overrides): several tiles per segment, ragged tails, F and H that
# are not powers of two
SMALL = {
    "c1": dict(),                                                  # full size (fp32)
    "c2": dict(T=384, H=512, E=16, k=4, F=384),
    "c3": dict(T=320, H=512, E=12, k=3, F=256, F_shared=384),
    "c4": dict(T=300, H=768, E=10, k=4, F=256, F_shared=640, layers=1),
    "c5": dict(T=520, H=512, E=4, k=2, F=1152),
}


def small_workload(key):
    cfg = W.CONFIGS[key]
    if SMALL[key]:
        cfg = W.scaled(cfg, **SMALL[key])
    return W.make_workload(cfg)


def run_layer(stack, wl, layer=0, X=None, Y0=None):
    from routed_expert_ffn_topk_gb300 import estream as es
    dev = _gpu.device()
    X = (wl.X if X is None else X).to(dev)
    lg = wl.logits[layer].to(dev)
    Y = torch.zeros(X.shape[0], wl.cfg.H, dtype=torch.float32, device=dev) if Y0 is None else Y0.to(dev).clone()
    stack.prefill(layer, X, lg, Y)
    torch.cuda.synchronize()
    assert es.get_device_error(stack.ctx) == es.OK
    return Y.cpu().numpy()


@pytest.mark.parametrize("key", sorted(SMALL))
@pytest.mark.parametrize("mode", ["resident", "paged"])
def test_layer_small_full_compare(key, mode):
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload(key)
    perm = W.random_permutation(wl.cfg.E, 11) if mode == "paged" else None
    st = BoundLayerStack(wl, mode=mode, perm=perm)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    ref = _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(y, ref, f"{key}/{mode}")


def test_layer_residual_accumulates():
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload("c2")
    st = BoundLayerStack(wl, mode="resident")
    try:
        A = torch.randn(wl.cfg.T, wl.cfg.H, generator=torch.Generator().manual_seed(9))
        y = run_layer(st, wl, Y0=A)
    finally:
        st.close()
    ref = _gpu.oracle_layer(wl, 0, wl.X, residual=A.double().numpy())
    _gpu.assert_y_close(y - A.numpy(), ref - A.double().numpy(), "residual")


@pytest.mark.parametrize("key,mode,form", [("c2", "resident", "auto"), ("c2", "resident", "pair"),
                                           ("c2", "paged", "auto"), ("c3", "paged", "auto"),
                                           ("c3", "resident", "single"), ("c5", "resident", "auto"),
                                           ("c5", "paged", "auto")])
def test_layer_full_size_sampled(key, mode, form):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.CONFIGS[key]
    wl = W.make_workload(cfg)
    f = {"auto": es.FFN_AUTO, "single": es.FFN_SINGLE, "pair": es.FFN_PAIR}[form]
    st = BoundLayerStack(wl, mode=mode, ffn_form=f)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    # a checked record in every (expert, 128-record block) of the route map
    rows = _gpu.rows_covering_mblocks(wl.logits[0].numpy(), cfg.k)
    ref = _gpu.oracle_layer(wl, 0, wl.X, rows=rows)
    _gpu.assert_y_close(y[rows], ref, f"{key}/{mode}/{form} {len(rows)} rows")


def test_layer_stack_chained_full_size():
    """Four Qwen-MoE-shaped layers through one P=16 arena; X_{l+1} = bf16(Y_l)
    with Y_l = X_l + MoE_l(X_l); each layer checked against the oracle fed the
    GPU's own X_l, on sampled rows."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.CONFIGS["c4"]
    wl = W.make_workload(cfg)
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode="paged")
    try:
        X = wl.X.to(dev)
        for l in range(cfg.layers):
            rows = _gpu.rows_covering_mblocks(wl.logits[l].numpy(), cfg.k)
            Y = X.float()
            st.prefill(l, X, wl.logits[l].to(dev), Y)
            torch.cuda.synchronize()
            assert es.get_device_error(st.ctx) == es.OK
            ref = _gpu.oracle_layer(wl, l, X.cpu(), rows=rows,
                                    residual=X.cpu().double().numpy())
            _gpu.assert_y_close(Y.cpu().numpy()[rows] - X.cpu().double().numpy()[rows],
                                ref - X.cpu().double().numpy()[rows], f"layer {l}")
            Xn = torch.empty_like(X)
            es.cast_f32_bf16(Y, Xn)
            assert torch.equal(Xn, Y.to(torch.bfloat16))   # RNE cast, bit for bit
            X = Xn
    finally:
        st.close()
