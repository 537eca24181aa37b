"""Degenerate and maximum shapes through the whole layer, in each form of the
fused kernel: a single expert (k = 1, every token routed to it), the largest
expert count and k the route build accepts (E = 1024, k = 32), one token, and
one n-block of F (F = 128)."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu
from tests.test_gpu_layer import run_layer

pytestmark = pytest.mark.gpu

SHAPES = {
    "single_expert": dict(T=200, H=256, E=1, k=1, F=256),
    "max_E_k": dict(T=40, H=256, E=1024, k=32, F=128),
    "one_token": dict(T=1, H=512, E=16, k=4, F=256),
    "one_n_block": dict(T=300, H=256, E=8, k=2, F=128),
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("form", ["single", "pair", "q4"])
def test_degenerate_shapes(shape, form):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.scaled(W.CONFIGS["c2"], **SHAPES[shape])
    wl = W.make_workload(cfg)
    kw = {"ffn_form": es.FFN_PAIR if form == "pair" else es.FFN_SINGLE}
    if form == "q4":
        kw["wdtype"] = es.Q4
    st = BoundLayerStack(wl, mode="resident", **kw)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    ref = _gpu.oracle_layer_q4(wl, 0, wl.X) if form == "q4" else _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(y, ref, f"{shape}/{form}")
