"""estream_moe_layer_prefill_residual: Y = A + MoE(X) with the residual rows
written by the route build (or, when T exceeds the rows its added CTAs cover,
by the first expert launch), against an explicit copy of A into Y followed by
the accumulating call (bit for bit in deterministic mode) and the oracle."""
import numpy as np
import pytest
import torch

from tests import _gpu
from tests.test_gpu_layer import small_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key,mode,q4", [("c2", "resident", False), ("c3", "paged", False),
                                         ("c2", "resident", True), ("c1", "resident", False)])
def test_residual_call(key, mode, q4):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload(key)
    dev = _gpu.device()
    ref = (_gpu.oracle_layer_q4(wl, 0, wl.X) if q4 else _gpu.oracle_layer(wl, 0, wl.X))
    # a residual on the scale of the MoE output, so that Y - A keeps its precision
    scale = float(np.abs(ref).mean())
    A_cpu = (torch.randn(wl.X.shape, generator=torch.Generator().manual_seed(17)) * scale).to(wl.X.dtype)
    st = BoundLayerStack(wl, mode=mode, deterministic=True, wdtype=es.Q4 if q4 else None)
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        A = A_cpu.to(dev)
        Y1 = A.float().clone()
        st.prefill(0, X, lg, Y1)
        Y2 = torch.full_like(Y1, float("nan"))   # every element must be written
        st.prefill(0, X, lg, Y2, residual=A)
        Y3 = torch.full_like(Y1, float("nan"))
        st.prefill(0, X, lg, Y3, residual=X)      # the residual stream itself
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        assert torch.equal(Y1.view(torch.int32), Y2.view(torch.int32))
    finally:
        st.close()
    Ac = A_cpu.double().numpy()
    _gpu.assert_y_close(Y2.cpu().numpy() - Ac, ref, f"residual A {key}/{mode}")
    # Y3 = X + MoE: compared with the oracle's Y including the same residual
    ref3 = (_gpu.oracle_layer_q4(wl, 0, wl.X) if q4 else None)
    if ref3 is None:
        ref3 = _gpu.oracle_layer(wl, 0, wl.X, residual=wl.X.double().numpy())
    else:
        ref3 = ref3 + wl.X.double().numpy()
    _gpu.assert_y_close(Y3.cpu().numpy(), ref3, f"residual X {key}/{mode}")


@pytest.mark.parametrize("T,E,k", [(4096, 300, 2), (100, 64, 8), (2500, 33, 3), (1, 8, 2)])
def test_residual_rows_bit_exact(T, E, k):
    """Residual rows at shapes that use every path of the route build's row
    writers: CTAs added for rows only (small T), top-k CTAs that also take rows
    (T = 4096: more chunks than added CTAs fit), ragged last chunks, one token,
    and E above 256 (the widest per-lane logit arrays). Bit for bit against a
    copy of A into Y followed by the accumulating call (deterministic mode)."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300 import workloads as W
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.scaled(W.CONFIGS["c2"], T=T, H=256, E=E, k=k, F=128, key_suffix=f"-resid{T}")
    wl = W.make_workload(cfg, seed=T + E)
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode="resident", deterministic=True)
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        A = torch.randn(X.shape, generator=torch.Generator().manual_seed(T), dtype=torch.float32)
        A = A.to(X.dtype).to(dev)
        Y1 = A.float().clone()
        st.prefill(0, X, lg, Y1)
        Y2 = torch.full_like(Y1, float("nan"))
        st.prefill(0, X, lg, Y2, residual=A)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        assert torch.equal(Y1.view(torch.int32), Y2.view(torch.int32))
    finally:
        st.close()


@pytest.mark.parametrize("mode", ["resident", "paged"])
def test_residual_rows_when_routing_times_out(mode):
    """At T = 4096 an expert launch writes the residual rows (more rows than
    the route build's added CTAs cover). When the route build's bounded
    barrier runs out (one CTA withholds its arrival) the route map is empty:
    resident, the routed launch still runs and writes the rows; paged, no
    group has work, no expert launch runs, and a copy kernel writes them. Y
    equals A bit for bit, the timeout is reported, and the next call is
    normal."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300 import workloads as W
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.scaled(W.CONFIGS["c2"], T=4096, H=256, E=8, k=2, F=128, key_suffix="-resid-timeout")
    wl = W.make_workload(cfg, seed=4242)
    dev = _gpu.device()
    kw = dict(G=2, B=2) if mode == "paged" else {}
    st = BoundLayerStack(wl, mode=mode, **kw)
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        A = torch.randn(X.shape, generator=torch.Generator().manual_seed(5), dtype=torch.float32)
        A = A.to(X.dtype).to(dev)
        es.inject_route_timeout(st.ctx)
        Y = torch.full((cfg.T, cfg.H), float("nan"), device=dev)
        st.prefill(0, X, lg, Y, residual=A)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.ERR_TIMEOUT
        assert torch.equal(Y.view(torch.int32), A.float().view(torch.int32))
        Y2 = torch.full_like(Y, float("nan"))
        st.prefill(0, X, lg, Y2, residual=A)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        y2 = Y2.cpu().numpy()
    finally:
        st.close()
    Ac = A.cpu().double().numpy()
    ref = _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(y2 - Ac, ref, f"T=4096 residual after a route timeout ({mode})")
