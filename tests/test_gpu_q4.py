"""4-bit experts (weight-only Q4_0-style blocks, decoded in the fused
kernel) against the oracle layer evaluated on the oracle's own dequantised
weights."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu
from tests.test_gpu_layer import run_layer, small_workload

pytestmark = pytest.mark.gpu


def _stack(wl, **kw):
    from routed_expert_ffn_topk_gb300 import estream as es
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    return BoundLayerStack(wl, wdtype=es.Q4, **kw)


@pytest.mark.parametrize("key", ["c2", "c3", "c4", "c5"])
@pytest.mark.parametrize("mode", ["resident", "paged"])
@pytest.mark.parametrize("form", ["auto", "pair"])
def test_q4_small_layers(key, mode, form):
    """Both forms of the 4-bit kernel: the single-SM one (the automatic
    choice) and the CTA-pair one, in which each SM streams and expands half
    of every packed weight tile."""
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload(key)
    perm = W.random_permutation(wl.cfg.E, 5) if mode == "paged" else None
    f = es.FFN_PAIR if form == "pair" else es.FFN_AUTO
    st = _stack(wl, mode=mode, perm=perm, ffn_form=f)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    ref = _gpu.oracle_layer_q4(wl, 0, wl.X)
    _gpu.assert_y_close(y, ref, f"q4 {key}/{mode}/{form}")


@pytest.mark.parametrize("mode,deterministic", [("resident", False), ("paged", False),
                                                ("resident", True)])
def test_q4_pair_segment_edges(mode, deterministic):
    """The 4-bit pair form on expert segments of 0, 1, 127, 128, 129, 255, 256,
    257, 383 and 512 records (pair tiles with an empty, partial or full second
    half; this form has no half tiles), against the oracle."""
    from routed_expert_ffn_topk_gb300 import estream as es
    from tests.test_gpu_pair import edge_workload
    wl, _ = edge_workload()
    kw = dict(G=4, B=2) if mode == "paged" else {}
    st = _stack(wl, mode=mode, ffn_form=es.FFN_PAIR, deterministic=deterministic, **kw)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    _gpu.assert_y_close(y, _gpu.oracle_layer_q4(wl, 0, wl.X),
                        f"q4 pair edges/{mode}/det={deterministic}")


def test_q4_deterministic_and_arena_independent():
    """Deterministic mode: bit-identical Y from a resident arena and from a
    small paged one."""
    wl = small_workload("c3")
    ys = []
    for kw in (dict(mode="resident"), dict(mode="paged", G=2, B=2)):
        st = _stack(wl, deterministic=True, **kw)
        try:
            ys.append(run_layer(st, wl))
        finally:
            st.close()
    assert np.array_equal(ys[0].view(np.uint32), ys[1].view(np.uint32))
    _gpu.assert_y_close(ys[0], _gpu.oracle_layer_q4(wl, 0, wl.X), "q4 deterministic")


@pytest.mark.parametrize("mode", ["resident", "paged"])
def test_q4_full_size_sampled(mode):
    cfg = W.CONFIGS["c2"]
    wl = W.make_workload(cfg)
    st = _stack(wl, mode=mode)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    rows = _gpu.rows_covering_mblocks(wl.logits[0].numpy(), cfg.k)   # every m-block
    ref = _gpu.oracle_layer_q4(wl, 0, wl.X, rows=rows)
    _gpu.assert_y_close(y[rows], ref, f"q4 c2/{mode} {len(rows)} rows")


@pytest.mark.parametrize("mode", ["resident", "paged"])
def test_q4_pair_full_size(mode):
    """The OLMoE-shaped layer at full size in the 4-bit pair form, on rows
    covering every m-block of the route map."""
    from routed_expert_ffn_topk_gb300 import estream as es
    cfg = W.CONFIGS["c2"]
    wl = W.make_workload(cfg)
    st = _stack(wl, mode=mode, ffn_form=es.FFN_PAIR)
    try:
        st.poison()
        y = run_layer(st, wl)
    finally:
        st.close()
    rows = _gpu.rows_covering_mblocks(wl.logits[0].numpy(), cfg.k)
    ref = _gpu.oracle_layer_q4(wl, 0, wl.X, rows=rows)
    _gpu.assert_y_close(y[rows], ref, f"q4 pair c2/{mode} {len(rows)} rows")
