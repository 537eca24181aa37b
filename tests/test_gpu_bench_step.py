"""The step bench.py times, at full size and in its launch configuration:
experts resident, the automatic kernel form, the residual entry point with
A = X (Y = X + MoE(X)), replayed from a CUDA graph. The graph is replayed
twice on different inputs copied into its buffers, with the workspace
poisoned (NaN) before each replay, and each replay is compared with the
oracle's Eq. 2 (residual included) on token rows that put a checked record
in every (expert, 128-record block) of the route map."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu

pytestmark = pytest.mark.gpu


def _capture(fn):
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        for _ in range(2):
            fn()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


@pytest.mark.parametrize("key", ["c2", "c3", "c5"])
def test_bench_step_full_size(key):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.CONFIGS[key]
    wl = W.make_workload(cfg, seed=W.CONFIG_SEEDS[key])
    dev = _gpu.device()
    st = BoundLayerStack(wl, mode="resident")
    try:
        X = wl.X.to(dev).clone()
        lg = wl.logits[0].to(dev).clone()
        Y = torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev)
        g = _capture(lambda: st.prefill(0, X, lg, Y, residual=X))
        for n, seed in enumerate([None, W.CONFIG_SEEDS[key] + 200]):
            if seed is None:
                X_cpu, lg_cpu = wl.X, wl.logits[0]
            else:
                other = W.make_workload(cfg, seed=seed, weights=False)
                X_cpu, lg_cpu = other.X, other.logits[0]
            X.copy_(X_cpu.to(dev))
            lg.copy_(lg_cpu.to(dev))
            Y.fill_(float("nan"))
            st.poison()
            g.replay()
            torch.cuda.synchronize()
            assert es.get_device_error(st.ctx) == es.OK
            y = Y.cpu().numpy()
            assert np.isfinite(y).all()
            rows = _gpu.rows_covering_mblocks(lg_cpu.numpy(), cfg.k)
            A = X_cpu.double().numpy()
            wl_n = W.Workload(cfg, [lg_cpu], X_cpu, wl.layers)
            ref = _gpu.oracle_layer(wl_n, 0, X_cpu, rows=rows, residual=A)
            # the tolerance applies to the MoE term; the residual is exact in fp32
            _gpu.assert_y_close(y[rows] - A[rows], ref - A[rows],
                                f"{key} bench step replay {n} ({len(rows)} rows)")
        del g
    finally:
        st.close()


def test_bench_step_layer_stack_full_size():
    """The four-layer Qwen-shaped step as bench.py runs it: one resident
    arena per layer, X_{l+1} = bf16(Y_l) between layers, the whole step
    replayed from one CUDA graph with every context's workspace poisoned
    first; each layer is checked against the oracle fed the GPU's own X_l on
    rows covering every m-block of that layer's route map."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.CONFIGS["c4"]
    wl = W.make_workload(cfg)
    dev = _gpu.device()
    L = cfg.layers
    one = cfg.__class__(**{**cfg.__dict__, "layers": 1})
    stacks = [BoundLayerStack(W.Workload(one, [wl.logits[l]], wl.X, [wl.layers[l]]), mode="resident")
              for l in range(L)]
    try:
        Xs = [wl.X.to(dev)] + [torch.empty(cfg.T, cfg.H, dtype=torch.bfloat16, device=dev)
                               for _ in range(L - 1)]
        lgs = [wl.logits[l].to(dev) for l in range(L)]
        Ys = [torch.empty(cfg.T, cfg.H, dtype=torch.float32, device=dev) for _ in range(L)]

        def step():
            for l in range(L):
                stacks[l].prefill(0, Xs[l], lgs[l], Ys[l], residual=Xs[l])
                if l + 1 < L:
                    es.cast_f32_bf16(Ys[l], Xs[l + 1])

        g = _capture(step)
        for y_ in Ys:
            y_.fill_(float("nan"))
        for s_ in stacks:
            s_.poison()
        g.replay()
        torch.cuda.synchronize()
        for s_ in stacks:
            assert es.get_device_error(s_.ctx) == es.OK
        for l in range(L):
            X_cpu = Xs[l].cpu()
            y = Ys[l].cpu().numpy()
            assert np.isfinite(y).all()
            rows = _gpu.rows_covering_mblocks(wl.logits[l].numpy(), cfg.k)
            A = X_cpu.double().numpy()
            ref = _gpu.oracle_layer(wl, l, X_cpu, rows=rows, residual=A)
            _gpu.assert_y_close(y[rows] - A[rows], ref - A[rows],
                                f"c4 stack layer {l} ({len(rows)} rows)")
            if l + 1 < L:
                assert torch.equal(Xs[l + 1].cpu(), Ys[l].cpu().to(torch.bfloat16))
        del g
    finally:
        for s_ in stacks:
            s_.close()
