"""A resident layer call (route build + fused expert kernel, no host
synchronisation) captured into a CUDA graph replays to the same Y as the
eager call, for each form of the fused kernel and for 4-bit experts."""
import numpy as np
import pytest
import torch

from tests import _gpu
from tests.test_gpu_layer import small_workload

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key,form,q4", [("c2", "single", False), ("c3", "pair", False),
                                         ("c2", "single", True)])
def test_layer_call_replays_from_cuda_graph(key, form, q4):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload(key)
    dev = _gpu.device()
    f = es.FFN_SINGLE if form == "single" else es.FFN_PAIR
    st = BoundLayerStack(wl, mode="resident", ffn_form=f, deterministic=True,
                         wdtype=es.Q4 if q4 else None)
    g = None
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        Y = torch.empty(wl.cfg.T, wl.cfg.H, dtype=torch.float32, device=dev)

        def call():
            Y.copy_(X)
            st.prefill(0, X, lg, Y)

        call()
        torch.cuda.synchronize()
        eager = Y.clone()
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            call()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            call()
        for _ in range(2):
            Y.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert es.get_device_error(st.ctx) == es.OK
            assert torch.equal(Y.view(torch.int32), eager.view(torch.int32))
    finally:
        g = None  # the graph records the context's events: release it first
        torch.cuda.synchronize()
        st.close()
    y = eager.cpu().numpy()
    ref = _gpu.oracle_layer_q4(wl, 0, wl.X) if q4 else _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(y - wl.X.float().numpy(), ref, f"graph {key}/{form}/q4={q4}")
