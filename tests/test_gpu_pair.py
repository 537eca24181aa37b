"""Both forms of the bf16 fused expert kernel -- 128-record tiles on one SM
and 256-record tiles on a cluster pair of SMs -- against the oracle, with
expert segments whose sizes sit on every tile edge of the pair form: empty,
one record, one short of, exactly at and one past 128, 256 and 384 records
(a pair tile whose second half is empty, partly filled or full)."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu
from tests.test_gpu_layer import run_layer, small_workload

pytestmark = pytest.mark.gpu

EDGE_COUNTS = [0, 1, 127, 128, 129, 255, 256, 257, 383, 512]


def edge_workload():
    """Top-1 routing with a fixed number of tokens per expert, tokens in a
    random order (so every segment gathers scattered rows)."""
    E = len(EDGE_COUNTS)
    T = sum(EDGE_COUNTS)
    cfg = W.scaled(W.CONFIGS["c2"], T=T, H=256, E=E, k=1, F=256)
    wl = W.make_workload(cfg)
    g = torch.Generator().manual_seed(21)
    expert_of = torch.cat([torch.full((n,), e, dtype=torch.int64) for e, n in enumerate(EDGE_COUNTS)])
    expert_of = expert_of[torch.randperm(T, generator=g)]
    lg = torch.randn(T, E, generator=g) * 0.1
    lg[torch.arange(T), expert_of] = 5.0
    return W.Workload(cfg, [lg], wl.X, wl.layers), expert_of


@pytest.mark.parametrize("form", ["single", "pair"])
@pytest.mark.parametrize("mode,deterministic", [("resident", False), ("paged", False),
                                                ("resident", True)])
def test_segment_edges(form, mode, deterministic):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl, expert_of = edge_workload()
    f = es.FFN_SINGLE if form == "single" else es.FFN_PAIR
    kw = dict(G=4, B=2) if mode == "paged" else {}
    st = BoundLayerStack(wl, mode=mode, ffn_form=f, deterministic=deterministic, **kw)
    try:
        out = es.route_build(wl.logits[0].to(_gpu.device()), 1, False)
        counts = (out["offsets"][1:wl.cfg.E + 1] - out["offsets"][:wl.cfg.E]).cpu().numpy()
        assert list(counts) == EDGE_COUNTS
        y = run_layer(st, wl)
    finally:
        st.close()
    ref = _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(y, ref, f"edges/{form}/{mode}/det={deterministic}")


@pytest.mark.parametrize("key", ["c2", "c3", "c4", "c5"])
@pytest.mark.parametrize("form", ["single", "pair"])
def test_small_layers_both_forms(key, form):
    """Every bf16 family's small shape (routed and shared experts) in each
    form, resident."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload(key)
    f = es.FFN_SINGLE if form == "single" else es.FFN_PAIR
    st = BoundLayerStack(wl, mode="resident", ffn_form=f)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    ref = _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(y, ref, f"{key}/{form}")


def test_forms_agree_closely():
    """The two forms compute the same tiles in the same K order; their Y may
    differ only by the order of the fp32 reductions into Y."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload("c5")
    ys = []
    for f in (es.FFN_SINGLE, es.FFN_PAIR):
        st = BoundLayerStack(wl, mode="resident", ffn_form=f, deterministic=True)
        try:
            ys.append(run_layer(st, wl))
        finally:
            st.close()
    d = np.abs(ys[0] - ys[1]).max() / np.abs(ys[0]).max()
    assert d <= 1e-5, d


def test_invalid_form_rejected():
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    wl = small_workload("c2")
    with pytest.raises(es.EStreamError) as ei:
        BoundLayerStack(wl, mode="resident", ffn_form=3)
    assert ei.value.status == es.ERR_INVALID_ARG


def test_split_down_tiles():
    """Down tiles of at least 128 k-blocks (F >= 8192) run as two K halves
    that each add their partial product into Y; Y against the oracle on
    every element, and against the deterministic mode (whole down tiles,
    rows combined in a fixed order) within the fp32 summation order."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    cfg = W.scaled(W.CONFIGS["c5"], T=520, H=512, E=4, k=2, F=8192)
    wl = W.make_workload(cfg)
    ys = {}
    for det in (False, True):
        st = BoundLayerStack(wl, mode="resident", ffn_form=es.FFN_PAIR, deterministic=det)
        try:
            ys[det] = run_layer(st, wl)
        finally:
            st.close()
    ref = _gpu.oracle_layer(wl, 0, wl.X)
    _gpu.assert_y_close(ys[False], ref, "F=8192 split down tiles")
    d = np.abs(ys[False] - ys[True]).max() / np.abs(ys[True]).max()
    assert d <= 1e-5, d
