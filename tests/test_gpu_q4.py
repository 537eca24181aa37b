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
def test_q4_small_layers(key, mode):
    wl = small_workload(key)
    perm = W.random_permutation(wl.cfg.E, 5) if mode == "paged" else None
    st = _stack(wl, mode=mode, perm=perm)
    try:
        y = run_layer(st, wl)
    finally:
        st.close()
    ref = _gpu.oracle_layer_q4(wl, 0, wl.X)
    _gpu.assert_y_close(y, ref, f"q4 {key}/{mode}")


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


def test_q4_rejects_pair_form():
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    with pytest.raises(es.EStreamError) as ei:
        _stack(wl, mode="resident", ffn_form=es.FFN_PAIR)
    assert ei.value.status == es.ERR_UNSUPPORTED
