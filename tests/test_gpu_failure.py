"""Failure detection on the GPU without a fault: the route build's bounded
grid barrier. One CTA withholds its arrival (a test hook), the others' wait
runs out after 1 s, the call leaves an empty route map and the error is
reported through estream_get_device_error; the next call is normal."""
import pytest
import torch

from tests import _gpu
from tests.test_gpu_layer import small_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("mode,deterministic", [("resident", False), ("paged", False),
                                                ("resident", True)])
def test_route_barrier_timeout_is_reported(mode, deterministic):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload("c2")
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode=mode, deterministic=deterministic)
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        Y_ref = torch.full((X.shape[0], wl.cfg.H), float("nan"), device=dev)
        st.prefill(0, X, lg, Y_ref, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK

        es.inject_route_timeout(st.ctx)
        Y = torch.full_like(Y_ref, float("nan"))
        if mode == "paged":
            es.arena_invalidate(st.ctx)
        st.prefill(0, X, lg, Y, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.ERR_TIMEOUT
        if not deterministic:
            # no routed expert ran: Y holds the residual rows only
            assert torch.equal(Y, X.float())

        Y2 = torch.full_like(Y_ref, float("nan"))
        st.prefill(0, X, lg, Y2, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        if deterministic:
            assert torch.equal(Y2.view(torch.int32), Y_ref.view(torch.int32))
        else:
            scale = float(Y_ref.abs().max())
            assert float((Y2 - Y_ref).abs().max()) <= 1e-5 * scale
    finally:
        st.close()


@pytest.mark.parametrize("form", ["single", "pair", "q4", "q4pair"])
def test_expert_kernel_timeout_is_reported(form):
    """The expert kernels' bounded waits: a call that runs the down tiles
    without their gate/up tiles (a test hook) waits 2 s for m-block counters
    that never fill; every CTA stops, drains and frees its tensor memory, the
    timeout is reported, and the next call is normal."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload("c2")
    dev = _gpu.device()
    kw = {"ffn_form": es.FFN_PAIR} if form == "pair" else (
        {"wdtype": es.Q4} if form == "q4" else (
            {"wdtype": es.Q4, "ffn_form": es.FFN_PAIR} if form == "q4pair" else
            {"ffn_form": es.FFN_SINGLE}))
    st = BoundLayerStack(wl, mode="resident", deterministic=True, **kw)
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        Y_ref = torch.full((X.shape[0], wl.cfg.H), float("nan"), device=dev)
        st.prefill(0, X, lg, Y_ref, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK

        es.inject_expert_timeout(st.ctx)
        Y = torch.full_like(Y_ref, float("nan"))
        st.prefill(0, X, lg, Y, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.ERR_TIMEOUT

        Y2 = torch.full_like(Y_ref, float("nan"))
        st.prefill(0, X, lg, Y2, residual=X)
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        assert torch.equal(Y2.view(torch.int32), Y_ref.view(torch.int32))
    finally:
        st.close()
