"""Arena pager and residency protocol (section 3.3 / 3.4 of the EStream
paper): results independent of arena size and storage order, every bank
published before use and released before refill, empty groups skipped, host
fault injection."""
import numpy as np
import pytest
import torch

from routed_expert_ffn_topk_gb300 import workloads as W
from tests import _gpu
from tests.test_gpu_layer import run_layer, small_workload

pytestmark = pytest.mark.gpu


def _stack(wl, **kw):
    from routed_expert_ffn_topk_gb300.layer import BoundLayerStack
    return BoundLayerStack(wl, **kw)


def test_deterministic_mode_bit_identical_across_arenas():
    """With the fixed-order combine, Y does not depend on the arena size,
    the group size or the storage order pi, resident or paged."""
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    E = wl.cfg.E
    ys = []
    for mode, G, B, seed, sched in [("resident", 4, None, None, es.SCHED_AFTER_ROUTING),
                                    ("paged", 4, 2, 1, es.SCHED_AFTER_ROUTING),
                                    ("paged", 2, 3, 2, es.SCHED_PREFETCH),
                                    ("paged", 16, 1, 3, es.SCHED_AFTER_ROUTING),
                                    ("paged", 3, 2, 4, es.SCHED_PREFETCH)]:
        perm = None if seed is None else W.random_permutation(E, seed)
        st = _stack(wl, mode=mode, G=G, B=B, perm=perm, deterministic=True, schedule=sched)
        try:
            ys.append(run_layer(st, wl))
        finally:
            st.close()
    for y in ys[1:]:
        np.testing.assert_array_equal(y, ys[0])
    _gpu.assert_y_close(ys[0], _gpu.oracle_layer(wl, 0, wl.X), "deterministic")


def _check_trace(trace, layer):
    """Per bank: Available -> Filling -> Ready -> (InUse -> Available | Available)."""
    state = {}
    content = {}
    for bank, l, g, s in trace:
        prev = state.get(bank, 0)
        if s == 1:
            assert prev == 0, f"bank {bank} filled while {prev}"
        elif s == 2:
            assert prev == 1 and content[bank] == (l, g)
        elif s == 3:
            assert prev == 2 and content[bank] == (l, g), f"bank {bank} used before Ready"
        elif s == 0:
            assert prev in (2, 3)
        content[bank] = (l, g)
        state[bank] = s
    assert all(v == 0 for v in state.values()), "a bank was left in use"


@pytest.mark.parametrize("sched", [0, 1])
def test_residency_protocol_and_bytes(sched):
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    cfg = wl.cfg
    # make expert storage group 1 (positions 4..7 under identity pi) unused
    lg = wl.logits[0].clone()
    lg[:, 4:8] = -30.0
    wl.logits[0] = lg
    st = _stack(wl, mode="paged", G=4, B=2, schedule=sched)
    try:
        es.set_timing(st.ctx, True)
        y = run_layer(st, wl)
        stats = es.last_stats(st.ctx)
        trace = es.residency_trace(st.ctx)
    finally:
        st.close()
    _check_trace(trace, 0)
    W_e = 3 * cfg.H * cfg.F * 2
    n_groups = cfg.E // 4
    loaded = stats["groups_loaded"]
    assert stats["groups_skipped"] == 1 and loaded == n_groups - 1
    prefetch_extra = 1 if sched == 1 else 0   # group 1 is among the first B=2 prefetched
    assert stats["h2d_bytes"] == (loaded + prefetch_extra) * 4 * W_e
    used = {g for (_, _, g, s) in trace if s == 3}
    assert 1 not in used
    _gpu.assert_y_close(y, _gpu.oracle_layer(wl, 0, wl.X), "skip")


def test_pager_fault_injection_leaves_context_usable():
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    st = _stack(wl, mode="paged", G=4, B=2)
    try:
        es.inject_pager_fault(st.ctx, 0, 2)
        dev = _gpu.device()
        Y = torch.zeros(wl.cfg.T, wl.cfg.H, device=dev)
        with pytest.raises(es.EStreamError) as ei:
            st.prefill(0, wl.X.to(dev), wl.logits[0].to(dev), Y)
        assert ei.value.status == es.ERR_PAGER
        es.inject_pager_fault(st.ctx, 0, -1)
        y = run_layer(st, wl)
    finally:
        st.close()
    _gpu.assert_y_close(y, _gpu.oracle_layer(wl, 0, wl.X), "after fault")


def test_capacity_and_argument_errors():
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    st = _stack(wl, mode="resident")
    dev = _gpu.device()
    try:
        X = torch.zeros(wl.cfg.T + 1, wl.cfg.H, dtype=torch.bfloat16, device=dev)
        lg = torch.zeros(wl.cfg.T + 1, wl.cfg.E, device=dev)
        Y = torch.zeros(wl.cfg.T + 1, wl.cfg.H, device=dev)
        with pytest.raises(es.EStreamError) as ei:
            st.prefill(0, X, lg, Y)
        assert ei.value.status == es.ERR_CAPACITY
        with pytest.raises(es.EStreamError) as ei:
            st.prefill(0, X[:4], lg[:4], Y[:4], k=wl.cfg.k + 1)
        assert ei.value.status == es.ERR_CAPACITY
        with pytest.raises(es.EStreamError) as ei:
            st.prefill(3, X[:4], lg[:4], Y[:4])
        assert ei.value.status == es.ERR_INVALID_ARG
    finally:
        st.close()


def test_ragged_token_counts_reuse_one_context():
    """T below T_max, including T=1 and T not a multiple of the tile."""
    wl = small_workload("c2")
    st = _stack(wl, mode="paged", G=4, B=2)
    try:
        for T in (1, 7, 129, wl.cfg.T):
            X = wl.X[:T].contiguous()
            sub = W.Workload(wl.cfg, [wl.logits[0][:T].contiguous()], X, wl.layers)
            y = run_layer(st, sub, X=X)
            ref = _gpu.oracle_layer(sub, 0, X)
            _gpu.assert_y_close(y, ref, f"T={T}")
    finally:
        st.close()


@pytest.mark.parametrize("Q", [1, 2])
def test_pipeline_trace_matches_max_plus_model(Q):
    """Per-group read/execution times recorded by the pager follow the
    max-plus recurrence of section 3.4 (Eq. 5): event order a <= d <= s <= f,
    no execution before its read ends, no bank refilled before its previous
    group finished, and the model fed the measured L = d - a, X = f - s
    predicts the measured completion."""
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    st = _stack(wl, mode="paged", G=2, B=2, Q=Q)
    try:
        es.set_timing(st.ctx, True)
        y = run_layer(st, wl)
        adsf, t_ne = es.pipeline_trace(st.ctx)
        stats = es.last_stats(st.ctx)
    finally:
        st.close()
    _gpu.assert_y_close(y, _gpu.oracle_layer(wl, 0, wl.X), f"Q={Q}")
    K = len(adsf)
    assert K == stats["groups_loaded"] and K >= 2
    a, d, s, f = adsf.T
    eps = 1e-3
    assert np.all(a <= d + eps) and np.all(d <= s + eps) and np.all(s <= f + eps)
    assert np.all(s[1:] >= f[:-1] - eps)           # one execution at a time
    assert np.all(a[2:] >= f[:-2] - eps)           # bank reuse waits for release (b = 2)
    L, X = d - a, f - s
    t_model, _ = es.maxplus_pipeline(L, X, Q, 2, t_ne)
    assert abs(t_model - f[-1]) <= 0.25 * f[-1] + 0.05, (t_model, f[-1])


def test_stats_overlap_measures():
    """estream_last_stats's hidden_fraction and bubble_rate (section 3.4,
    Fig. 6): from the same calls' copy, execution and total times, within
    [0, 1]; a resident call copies nothing and hides nothing."""
    from routed_expert_ffn_topk_gb300 import estream as es
    wl = small_workload("c2")
    for mode in ("paged", "resident"):
        st = _stack(wl, mode=mode, G=4, B=2) if mode == "paged" else _stack(wl, mode=mode)
        try:
            run_layer(st, wl)
            es.reset_stats(st.ctx)
            es.set_timing(st.ctx, True)
            for _ in range(3):
                if mode == "paged":
                    es.arena_invalidate(st.ctx)
                run_layer(st, wl)
            s = es.last_stats(st.ctx)
        finally:
            st.close()
        t_io, t_tot = s["ms_io_busy"], s["ms_total"]
        t_ex = s["ms_route"] + s["ms_ffn"] + s["ms_shared"] + s["ms_combine"]
        assert 0.0 <= s["hidden_fraction"] <= 1.0 and 0.0 <= s["bubble_rate"] <= 1.0
        assert t_tot > 0
        want_b = min(1.0, max(0.0, 1.0 - max(t_io, t_ex) / t_tot))
        assert s["bubble_rate"] == pytest.approx(want_b, abs=1e-12)
        if mode == "paged":
            assert t_io > 0 and s["h2d_bytes"] > 0
            want_h = min(1.0, max(0.0, (t_io + t_ex - t_tot) / t_io))
            assert s["hidden_fraction"] == pytest.approx(want_h, abs=1e-12)
        else:
            assert t_io == 0 and s["hidden_fraction"] == 0.0
