"""Shared helpers of the GPU parity tests: tolerance checks against the
oracle, and device setup."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from routed_expert_ffn_topk_gb300 import workloads as W

# Tolerance for Y (bf16 weights/activations, fp32 accumulation): normwise
# max |dY| / max |Y_ref| <= 2e-2 and mean |dY| / mean |Y_ref| <= 1e-3.
MAX_REL = 2e-2
MEAN_REL = 1e-3


# Diagnostics of every comparison made in this session: (what, max_rel,
# mean_rel, elementwise max rel over the large entries), printed in pytest's
# terminal summary.
DIAGNOSTICS = []


def y_errors(y_gpu, y_ref):
    """Normwise max |dY| / max |Y_ref| and mean |dY| / mean |Y_ref|."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    d = np.abs(y_gpu - y_ref)
    return d.max() / np.abs(y_ref).max(), d.mean() / np.abs(y_ref).mean()


def elementwise_rel(y_gpu, y_ref):
    """Diagnostic beside the normwise bounds: the largest |dY| / |Y_ref| over
    the entries with |Y_ref| >= 0.1 mean |Y_ref| (the elementwise ratio is
    undefined near zero, so smaller entries are left out)."""
    y_gpu = np.asarray(y_gpu, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    a = np.abs(y_ref)
    big = a >= 0.1 * a.mean()
    if not big.any():
        return 0.0
    return float((np.abs(y_gpu - y_ref)[big] / a[big]).max())


def assert_y_close(y_gpu, y_ref, what=""):
    assert np.all(np.isfinite(y_gpu)), f"{what}: non-finite output"
    mx, mean = y_errors(y_gpu, y_ref)
    el = elementwise_rel(y_gpu, y_ref)
    DIAGNOSTICS.append((what, mx, mean, el))
    assert mx <= MAX_REL and mean <= MEAN_REL, \
        f"{what}: max_rel {mx:.3e} mean_rel {mean:.3e} (elementwise {el:.3e})"
    return mx, mean


def rows_covering_mblocks(logits, k, block=128):
    """Token rows such that every (expert, block of `block` records) of the
    route map holds at least one checked record: for each expert, its routes
    in ascending route index i = t*k + j (the order records take inside a
    slot) are cut into blocks, and the tokens of each block's first and last
    record are taken (the last one also covers a ragged tail). The top-k is
    taken as the largest logits, lower index first on ties."""
    lg = np.asarray(logits, dtype=np.float32)
    T, E = lg.shape
    order = np.lexsort((np.broadcast_to(np.arange(E), lg.shape), -lg), axis=1)
    ids = order[:, :k].reshape(-1)                       # route i = t*k + j
    rows = set()
    for e in range(E):
        routes = np.nonzero(ids == e)[0]                 # ascending i
        for b0 in range(0, len(routes), block):
            blk = routes[b0:b0 + block]
            rows.add(int(blk[0]) // k)
            rows.add(int(blk[-1]) // k)
    return np.array(sorted(rows), dtype=np.int64)


def oracle_layer(wl: W.Workload, layer: int, X_cpu, rows=None, residual=None):
    """Oracle routing + Eq. 2 for the listed rows of one layer."""
    cfg = wl.cfg
    lw = wl.layers[layer]
    ids, alpha = oracle.route_topk(wl.logits[layer].numpy(), cfg.k, cfg.renorm)
    shared = (lw.Sg, lw.Su, lw.Sd) if cfg.n_shared else None
    return oracle.moe_layer_rows(X_cpu, lw.Wg, lw.Wu, lw.Wd, ids, alpha, rows=rows,
                                 shared=shared, residual=residual)


def device():
    return torch.device("cuda", 0)


def q4_weights(lw):
    """The weights a 4-bit layer computes with, dequantised by the oracle:
    gate/up with bf16 block scales, down pre-scaled by 2^s with fp16 scales."""
    def gu(W):
        return np.stack([oracle.q4_dequantize(*oracle.q4_quantize(W[e], fp16=False)) for e in range(W.shape[0])])

    def dn(W):
        out = []
        for e in range(W.shape[0]):
            s = oracle.down_scale_exp(W[e])
            c, d = oracle.q4_quantize(W[e], fp16=True, scale_exp=s)
            out.append(oracle.q4_dequantize(c, d, scale_exp=s))
        return np.stack(out)
    shared = None
    if lw.Sg is not None:
        shared = (gu(lw.Sg), gu(lw.Su), dn(lw.Sd))
    return gu(lw.Wg), gu(lw.Wu), dn(lw.Wd), shared


def oracle_layer_q4(wl: W.Workload, layer: int, X_cpu, rows=None, dq=None):
    """Oracle routing + Eq. 2 with the dequantised 4-bit weights (X widened
    exactly to fp32)."""
    cfg = wl.cfg
    Wg, Wu, Wd, shared = dq if dq is not None else q4_weights(wl.layers[layer])
    ids, alpha = oracle.route_topk(wl.logits[layer].numpy(), cfg.k, cfg.renorm)
    Xf = torch.as_tensor(X_cpu).float().numpy()
    return oracle.moe_layer_rows(Xf, Wg, Wu, Wd, ids, alpha, rows=rows, shared=shared)
