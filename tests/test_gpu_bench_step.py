"""The step bench.py times, at full size and in its launch configuration:
experts resident, the automatic kernel form, the residual entry point with
A = X (Y = X + MoE(X)), replayed from a CUDA graph. Seeded samples of token
rows are compared with the oracle's Eq. 2 including the residual."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("key", ["c2", "c3", "c5"])
def test_bench_step_full_size(key):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.CONFIGS[key]
    wl = W.make_workload(cfg, seed=W.CONFIG_SEEDS[key])
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode="resident")
    try:
        X = wl.X.to(dev)
        lg = wl.logits[0].to(dev)
        Y = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev)

        def step():
            st.prefill(0, X, lg, Y, residual=X)

        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for _ in range(2):
                step()
        torch.cuda.current_stream().wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step()
        torch.cuda.synchronize()
        Y.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert es.get_device_error(st.ctx) == es.OK
        y = Y.cpu().numpy()
        del g
    finally:
        st.close()
    assert np.isfinite(y).all()
    rows = W.sample_rows(cfg.T, 24 if cfg.H * cfg.F < 2e7 else 10, seed=5)
    A = wl.X.double().numpy()
    ref = _gpu.oracle_layer(wl, 0, wl.X, rows=rows.numpy(), residual=A)
    r = rows.numpy()
    # the tolerance applies to the MoE term; the residual is exact in fp32
    _gpu.assert_y_close(y[r] - A[r], ref - A[r], f"{key} bench step (graph replay) sampled")
