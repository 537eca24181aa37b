"""Pins of the CPU oracle to facts it does not compute itself.

Each ``pin_*`` function takes a loaded oracle library and raises
AssertionError when the oracle disagrees with something the pages or the
mathematics fix: a closed form, a textbook routine, brute force on a tiny
input, an invariant, or a hand-worked fixture under ``tests/golden/``.
They are plain functions so the mutation test can run them against oracle
builds with planted mistakes.
"""
from __future__ import annotations

import math
import os

import numpy as np

from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# exponential
# --------------------------------------------------------------------------

def pin_exp(lib):
    """Written exp vs fp64 exp: within one fp32 ulp on [-87, 0]; exp(0) = 1;
    0 below -87; non-decreasing."""
    xs = np.concatenate([np.linspace(-87.0, 0.0, 20001, dtype=np.float32),
                         np.float32([-1e-30, -1e-7, -0.5, -0.34657359, -0.34657358, -1.0, -86.99])])
    xs = np.sort(xs)
    e = np.array([lib.oracle_exp_f32(float(v)) for v in xs], dtype=np.float64)
    ref = np.exp(xs.astype(np.float64))
    ulp = np.spacing(ref.astype(np.float32)).astype(np.float64)
    err = np.abs(e - ref) / ulp
    assert err.max() <= 1.0, f"exp error {err.max():.3f} ulp"
    assert lib.oracle_exp_f32(0.0) == 1.0
    assert lib.oracle_exp_f32(-88.0) == 0.0 and lib.oracle_exp_f32(-1e4) == 0.0
    assert np.all(np.diff(e) >= 0.0), "exp not monotone"


# --------------------------------------------------------------------------
# router
# --------------------------------------------------------------------------

def _brute_topk(logits, k):
    T, E = logits.shape
    ids = np.zeros((T, k), dtype=np.int32)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))
        ids[t] = order[:k]
    return ids


def _softmax64(logits):
    l = logits.astype(np.float64)
    z = np.exp(l - l.max(axis=1, keepdims=True))
    return z / z.sum(axis=1, keepdims=True)


def pin_topk(lib):
    """Top-k ids equal a full sort by (logit desc, id asc); each token has k
    distinct ids; alpha equals the fp64 softmax within a few fp32 ulps, and
    the renormalised weights sum to 1."""
    rng = _rng(1)
    for (T, E, k) in [(37, 8, 2), (16, 64, 8), (9, 60, 4), (5, 5, 5), (11, 1, 1)]:
        lg = rng.standard_normal((T, E)).astype(np.float32)
        lg[0, :] = 0.25                       # all-equal row
        if E > 3:
            lg[1, 1] = lg[1, 3] = lg[1].max() + 1.0   # a tie at the top
        for renorm in (0, 1):
            ids, al = O.route_topk(lg, k, renorm, lib=lib)
            np.testing.assert_array_equal(ids, _brute_topk(lg, k))
            for t in range(T):
                assert len(set(ids[t].tolist())) == k
            p = _softmax64(lg)
            sel = np.take_along_axis(p, ids.astype(np.int64), axis=1)
            if renorm:
                sel = sel / sel.sum(axis=1, keepdims=True)
                s = al.astype(np.float64).sum(axis=1)
                assert np.all(np.abs(s - 1.0) <= 4 * k * 2.0 ** -24), s
            rel = np.abs(al.astype(np.float64) - sel) / sel
            assert rel.max() < 2.0 ** -20 + (E + k) * 2.0 ** -24, rel.max()
    # k == E without renormalisation: alpha is the whole softmax, summing to 1
    lg = rng.standard_normal((6, 16)).astype(np.float32)
    ids, al = O.route_topk(lg, 16, 0, lib=lib)
    assert np.all(np.abs(al.astype(np.float64).sum(axis=1) - 1.0) < 16 * 2.0 ** -23)
    # one logit per token: softmax of a single value is exactly 1
    ids, al = O.route_topk(rng.standard_normal((4, 1)).astype(np.float32), 1, 0, lib=lib)
    assert np.all(al == 1.0) and np.all(ids == 0)


def pin_topk_golden(lib):
    """Hand-worked router example (tests/golden/router_example.txt)."""
    fx = _read_golden("router_example.txt")
    lg = np.array(fx["logits"], dtype=np.float32).reshape(-1, int(fx["E"][0]))
    k = int(fx["k"][0])
    for renorm, key_ids, key_alpha in ((0, "ids", "alpha"), (1, "ids", "alpha_renorm")):
        ids, al = O.route_topk(lg, k, renorm, lib=lib)
        np.testing.assert_array_equal(ids.ravel(), np.array(fx[key_ids], dtype=np.int32))
        want = np.array(fx[key_alpha], dtype=np.float64)
        assert np.all(np.abs(al.ravel().astype(np.float64) - want) <= 2 * np.spacing(np.float32(want))), (al, want)


# --------------------------------------------------------------------------
# route map
# --------------------------------------------------------------------------

def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line or ":" not in line:
                continue
            key, vals = line.split(":", 1)
            out[key.strip()] = [float(v) if "." in v or "e" in v.lower() else int(v)
                                for v in vals.split()]
    return out


def _brute_csr(ids, E, P, phi):
    T, k = ids.shape
    R = T * k
    flat = ids.ravel()
    psi = np.array([(phi[e] if phi is not None else e) for e in flat], dtype=np.int64)
    psi[psi < 0] = P
    order = np.argsort(psi, kind="stable")
    counts = np.bincount(psi, minlength=P + 1)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    return offsets, (order // k).astype(np.int32), order.astype(np.int32), psi


def pin_csr(lib):
    """Route map equals a stable counting sort by slot (numpy stable argsort,
    bincount + cumsum) and satisfies the CSR invariants."""
    rng = _rng(2)
    for (T, E, k, P, mode) in [(40, 8, 2, 8, "identity"), (64, 16, 4, 6, "partial"),
                               (33, 60, 4, 60, "perm"), (7, 4, 4, 1, "partial"), (1, 3, 1, 3, "identity"),
                               (0, 4, 2, 4, "identity")]:
        lg = rng.standard_normal((T, E)).astype(np.float32)
        ids, _ = O.route_topk(lg, k, 0, lib=lib) if T > 0 else (np.zeros((0, k), np.int32), None)
        if mode == "identity":
            phi = None
        elif mode == "perm":
            phi = rng.permutation(E).astype(np.int32)
        else:
            slots = rng.permutation(P)
            phi = -np.ones(E, dtype=np.int32)
            chosen = rng.choice(E, size=min(P, E), replace=False)
            phi[chosen] = slots[:len(chosen)]
        offs, rt, rr = O.route_csr(ids, E, P, phi, lib=lib)
        bo, bt, br, psi = _brute_csr(ids, E, P, phi)
        np.testing.assert_array_equal(offs, bo)
        np.testing.assert_array_equal(rt, bt)
        np.testing.assert_array_equal(rr, br)
        R = T * k
        assert offs[0] == 0 and offs[-1] == R and np.all(np.diff(offs) >= 0)
        assert sorted(rr.tolist()) == list(range(R))
        for s in range(P + 1):
            seg = rr[offs[s]:offs[s + 1]]
            assert np.all(np.diff(seg) > 0), "records not in ascending route order"
            assert np.all(psi[seg] == s)


def pin_csr_golden(lib):
    """Hand-worked route map (tests/golden/route_map_example.txt)."""
    fx = _read_golden("route_map_example.txt")
    k, E, P = int(fx["k"][0]), int(fx["E"][0]), int(fx["P"][0])
    ids = np.array(fx["topk_ids"], dtype=np.int32).reshape(-1, k)
    phi = np.array(fx["phi"], dtype=np.int32)
    offs, rt, rr = O.route_csr(ids, E, P, phi, lib=lib)
    np.testing.assert_array_equal(offs, fx["offsets"])
    np.testing.assert_array_equal(rt, fx["rec_tok"])
    np.testing.assert_array_equal(rr, fx["rec_route"])


def pin_placement(lib):
    """Eq. 4 against the hand-worked fixture and against its definition's
    consequences: resident experts get distinct slots inside their bank."""
    fx = _read_golden("placement_example.txt")
    phi = O.grouped_placement(fx["perm"], int(fx["E"][0]), int(fx["G"][0]), fx["bank_of_group"], lib=lib)
    np.testing.assert_array_equal(phi, fx["phi"])
    rng = _rng(3)
    E, G = 60, 8
    perm = rng.permutation(E).astype(np.int32)
    nq = -(-E // G)
    bank = -np.ones(nq, dtype=np.int32)
    bank[rng.choice(nq, size=2, replace=False)] = [0, 1]
    phi = O.grouped_placement(perm, E, G, bank, lib=lib)
    res = phi[phi >= 0]
    assert len(set(res.tolist())) == len(res)
    for e in range(E):
        q = perm[e] // G
        if bank[q] < 0:
            assert phi[e] == -1
        else:
            assert bank[q] * G <= phi[e] < (bank[q] + 1) * G


# --------------------------------------------------------------------------
# expert FFN / layer
# --------------------------------------------------------------------------

def _small_layer(seed, T=12, H=32, E=4, F=24, k=2, renorm=0, n_shared=0, Fs=16):
    rng = _rng(seed)
    X = rng.standard_normal((T, H)).astype(np.float32)
    Wg = (0.3 * rng.standard_normal((E, F, H))).astype(np.float32)
    Wu = (0.3 * rng.standard_normal((E, F, H))).astype(np.float32)
    Wd = (0.3 * rng.standard_normal((E, H, F))).astype(np.float32)
    lg = rng.standard_normal((T, E)).astype(np.float32)
    shared = None
    if n_shared:
        shared = tuple((0.3 * rng.standard_normal(s)).astype(np.float32)
                       for s in ((n_shared, Fs, H), (n_shared, Fs, H), (n_shared, H, Fs)))
    return X, Wg, Wu, Wd, lg, shared


def _dense_layer64(X, Wg, Wu, Wd, ids, alpha, shared=None, residual=None):
    """Every token through every expert, masked by the top-k weights."""
    X = X.astype(np.float64)
    T = X.shape[0]
    E = Wg.shape[0]
    M = np.zeros((T, E))
    for t in range(T):
        for j in range(ids.shape[1]):
            M[t, ids[t, j]] += float(alpha[t, j])
    Y = np.zeros((T, Wd.shape[1])) if residual is None else residual.astype(np.float64).copy()
    for e in range(E):
        G = X @ Wg[e].astype(np.float64).T
        U = X @ Wu[e].astype(np.float64).T
        Z = (G / (1.0 + np.exp(-G)) * U) @ Wd[e].astype(np.float64).T
        Y += M[:, e:e + 1] * Z
    if shared is not None:
        for s in range(shared[0].shape[0]):
            G = X @ shared[0][s].astype(np.float64).T
            U = X @ shared[1][s].astype(np.float64).T
            Y += (G / (1.0 + np.exp(-G)) * U) @ shared[2][s].astype(np.float64).T
    return Y


def _rel(a, b):
    return np.abs(a - b).max() / max(np.abs(b).max(), 1e-300)


def pin_layer_dense(lib):
    """Eq. 2 evaluated per route equals the dense masked evaluation."""
    for seed, kw in ((10, {}), (11, dict(renorm=1, k=3)), (12, dict(n_shared=2)),
                     (13, dict(T=5, E=1, k=1))):
        X, Wg, Wu, Wd, lg, shared = _small_layer(seed, **kw)
        k = kw.get("k", 2)
        ids, al = O.route_topk(lg, k, kw.get("renorm", 0), lib=lib)
        Y = O.moe_layer_rows(X, Wg, Wu, Wd, ids, al, shared=shared, lib=lib)
        Yd = _dense_layer64(X, Wg, Wu, Wd, ids, al, shared)
        assert _rel(Y, Yd) < 1e-12, _rel(Y, Yd)
        rows = np.array([kw.get("T", 12) - 1, 0, 2], dtype=np.int32)
        Ys = O.moe_layer_rows(X, Wg, Wu, Wd, ids, al, rows=rows, shared=shared, lib=lib)
        np.testing.assert_array_equal(Ys, Y[rows])


def pin_layer_textbook(lib):
    """E = 1, k = 1 reduces to a dense SwiGLU FFN (torch silu + matmul, fp64)."""
    import torch
    X, Wg, Wu, Wd, lg, _ = _small_layer(20, T=9, E=1, k=1)
    ids, al = O.route_topk(lg, 1, 0, lib=lib)
    assert np.all(al == 1.0)
    Y = O.moe_layer_rows(X, Wg, Wu, Wd, ids, al, lib=lib)
    x = torch.from_numpy(X).double()
    ref = (torch.nn.functional.silu(x @ torch.from_numpy(Wg[0]).double().T)
           * (x @ torch.from_numpy(Wu[0]).double().T)) @ torch.from_numpy(Wd[0]).double().T
    assert _rel(Y, ref.numpy()) < 1e-12


def pin_layer_special(lib):
    """W_g = 0 gives Y = A exactly (SiLU(0) = 0); doubling W_d doubles Y
    exactly; a permutation of the hidden neurons changes only summation
    order; a residual adds; bf16 inputs equal their exact fp32 widening."""
    import torch
    X, Wg, Wu, Wd, lg, _ = _small_layer(30)
    ids, al = O.route_topk(lg, 2, 0, lib=lib)
    A = _rng(31).standard_normal((X.shape[0], X.shape[1]))
    Y0 = O.moe_layer_rows(X, np.zeros_like(Wg), Wu, Wd, ids, al, residual=A, lib=lib)
    np.testing.assert_array_equal(Y0, A)
    Y = O.moe_layer_rows(X, Wg, Wu, Wd, ids, al, lib=lib)
    Y2 = O.moe_layer_rows(X, Wg, Wu, 2 * Wd, ids, al, lib=lib)
    np.testing.assert_array_equal(Y2, 2 * Y)
    sig = _rng(32).permutation(Wg.shape[1])
    Yp = O.moe_layer_rows(X, Wg[:, sig], Wu[:, sig], Wd[:, :, sig], ids, al, lib=lib)
    assert _rel(Yp, Y) < 1e-13
    YA = O.moe_layer_rows(X, Wg, Wu, Wd, ids, al, residual=A, lib=lib)
    assert _rel(YA - A, Y) < 1e-13
    tb = lambda a: torch.from_numpy(a).to(torch.bfloat16)
    Yb = O.moe_layer_rows(tb(X), tb(Wg), tb(Wu), tb(Wd), ids, al, lib=lib)
    wide = lambda a: tb(a).to(torch.float32).numpy()
    Yf = O.moe_layer_rows(wide(X), wide(Wg), wide(Wu), wide(Wd), ids, al, lib=lib)
    np.testing.assert_array_equal(Yb, Yf)


# --------------------------------------------------------------------------
# pipeline model
# --------------------------------------------------------------------------

def pin_maxplus(lib):
    """Eq. 5 against a hand-worked fixture and closed forms: with unlimited
    banks and one read in flight it is the two-machine flow shop
    max_k (sum_{j<=k} L_j + sum_{j>=k} X_j); with one bank everything is
    serial, sum_k (L_k + X_k); with unlimited reads and banks every read
    starts at 0; more banks or reads never make it slower."""
    fx = _read_golden("maxplus_example.txt")
    t, adsf = O.maxplus(fx["L"], fx["X"], int(fx["q"][0]), int(fx["b"][0]), fx["T_ne"][0], lib=lib)
    for col, key in enumerate("adsf"):
        np.testing.assert_array_equal(adsf[:, col], fx[key])
    assert t == fx["f"][-1]
    rng = _rng(4)
    for K in (1, 2, 5, 17):
        L = rng.uniform(0.1, 3.0, K).round(3)
        X = rng.uniform(0.1, 3.0, K).round(3)
        flow = max(L[:k + 1].sum() + X[k:].sum() for k in range(K))
        t, _ = O.maxplus(L, X, 1, K + 5, 0.0, lib=lib)
        assert abs(t - flow) < 1e-9, (t, flow)
        t1, _ = O.maxplus(L, X, 1, 1, 0.0, lib=lib)
        assert abs(t1 - (L.sum() + X.sum())) < 1e-9
        tp, adsf = O.maxplus(L, X, K + 5, K + 5, 0.0, lib=lib)
        assert np.all(adsf[:, 0] == 0.0)
        np.testing.assert_allclose(adsf[:, 1], L)
        # no bank limit and every read done before the non-expert work ends:
        # execution is one serial run starting at T_ne
        tn, adsf = O.maxplus(L, X, 1, K + 5, 100.0, lib=lib)
        assert np.all(adsf[:, 2] >= 100.0) and abs(tn - (100.0 + X.sum())) < 1e-9
        prev = None
        for b in range(1, K + 3):
            tb, _ = O.maxplus(L, X, 2, b, 0.5, lib=lib)
            assert prev is None or tb <= prev + 1e-12
            prev = tb
        assert O.maxplus(L, X, 2, 3, 0.0, lib=lib)[0] <= O.maxplus(L, X, 1, 3, 0.0, lib=lib)[0] + 1e-12


# --------------------------------------------------------------------------
# router logits
# --------------------------------------------------------------------------

def _bf16_bits(a):
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _bf16_widen(b):
    return (b.astype(np.uint32) << 16).view(np.float32)


def pin_router(lib):
    """Router logits l = X W_r^T against exact integer arithmetic (small
    integer inputs, where every fp64 partial sum is exact), numpy's fp64
    matmul on random inputs (equal up to rounding order), a one-hot W_r (each
    expert reads one input feature, exactly), and bf16 inputs equal to their
    fp32 widening."""
    rng = _rng(11)
    for T, H, E in ((1, 1, 1), (3, 7, 5), (9, 64, 12), (4, 5, 9)):
        Xi = rng.integers(-8, 9, (T, H))
        Wi = rng.integers(-8, 9, (E, H))
        got = O.router_logits(Xi.astype(np.float32), Wi.astype(np.float32), lib=lib)
        exact = np.array([[sum(int(Xi[t, h]) * int(Wi[e, h]) for h in range(H)) for e in range(E)]
                          for t in range(T)], dtype=np.float64)
        np.testing.assert_array_equal(got, exact)
    X = rng.standard_normal((17, 96)).astype(np.float32)
    W = rng.standard_normal((10, 96)).astype(np.float32)
    got = O.router_logits(X, W, lib=lib)
    ref = X.astype(np.float64) @ W.astype(np.float64).T
    scale = np.abs(X).astype(np.float64) @ np.abs(W).astype(np.float64).T
    assert np.all(np.abs(got - ref) <= 1e-13 * scale)
    cols = rng.integers(0, 96, 10)
    onehot = np.zeros((10, 96), dtype=np.float32)
    onehot[np.arange(10), cols] = 1.0
    np.testing.assert_array_equal(O.router_logits(X, onehot, lib=lib), X[:, cols].astype(np.float64))
    Xb, Wb = _bf16_bits(X), _bf16_bits(W)
    np.testing.assert_array_equal(O.router_logits(Xb, Wb, lib=lib),
                                  O.router_logits(_bf16_widen(Xb), _bf16_widen(Wb), lib=lib))


# --------------------------------------------------------------------------
# 4-bit expert weights
# --------------------------------------------------------------------------

def pin_q4_golden(lib):
    """The hand-worked blocks of tests/golden/q4_block_example.txt, in both
    operand types (every scale there is exact in bf16 and fp16)."""
    fx = _read_golden("q4_block_example.txt")
    A = np.array([((j % 16) - 8) / 8.0 for j in range(32)], dtype=np.float32)
    B = np.zeros(32, dtype=np.float32)
    B[:6] = np.array(fx["B_x"], dtype=np.float32)
    C = np.zeros(32, dtype=np.float32)
    for fp16 in (False, True):
        codes, d = O.q4_quantize(np.stack([A, B, C]), fp16=fp16, lib=lib)
        for row, key in enumerate("ABC"):
            assert d[row, 0] == np.float32(fx[key + "_d"][0]), (key, d[row, 0])
            np.testing.assert_array_equal(codes[row], fx[key + "_q"])
        w = O.q4_dequantize(codes, d, lib=lib)
        np.testing.assert_array_equal(w[0], A)          # block A lies on its grid
        np.testing.assert_array_equal(w[2], C)
    assert O.down_scale_exp(np.array([[0.77, -0.5]], dtype=np.float32), lib=lib) == fx["s_for_0.77"][0]
    assert O.down_scale_exp(np.array([[-1.0, 0.25]], dtype=np.float32), lib=lib) == fx["s_for_1.0"][0]


def pin_q4_properties(lib):
    """Random blocks: every element whose code is not clamped lies within d/2
    of its dequantised value; codes in 0..15 and the largest element within
    8 |d - m/-8| of -8 d; a block already on a 5-bit grid is reproduced
    exactly; scaling a block by 2^k scales d by 2^k and keeps the codes;
    negating it negates d and keeps the codes; the pre-scale 2^s of a down
    plane is undone by the dequantiser."""
    rng = _rng(12)
    W = (rng.standard_normal((16, 128)) * 0.02).astype(np.float32)
    for fp16 in (False, True):
        codes, d = O.q4_quantize(W, fp16=fp16, lib=lib)
        assert codes.max() <= 15
        w = O.q4_dequantize(codes, d, lib=lib).astype(np.float64)
        dd = np.repeat(np.abs(d.astype(np.float64)), 32, axis=1)
        inner = (codes > 0) & (codes < 15)
        assert np.all(np.abs(w - W)[inner] <= dd[inner] / 2 * (1 + 1e-6))
        blocks = W.reshape(16, 4, 32)
        m = np.take_along_axis(blocks, np.abs(blocks).argmax(axis=2)[..., None], axis=2)[..., 0]
        assert np.all(np.abs(m / -8 - d) <= np.abs(m / -8) * 2.0 ** -5 * (1 + 1e-6))
        c2, d2 = O.q4_quantize(W * 4, fp16=fp16, lib=lib)
        np.testing.assert_array_equal(c2, codes)
        np.testing.assert_array_equal(d2, d * 4)
        c3, d3 = O.q4_quantize(-W, fp16=fp16, lib=lib)
        np.testing.assert_array_equal(c3, codes)
        np.testing.assert_array_equal(d3, -d)
    grid_d = np.float32(-1.0625 * 2.0 ** -6)                 # 5 significant bits
    q = rng.integers(0, 16, (2, 32))
    q[:, 0] = 0                                               # the block maximum is -8 d
    G = ((q - 8) * grid_d).astype(np.float32)
    cg, dg = O.q4_quantize(G, fp16=False, lib=lib)
    np.testing.assert_array_equal(cg, q)
    np.testing.assert_array_equal(O.q4_dequantize(cg, dg, lib=lib), G)
    s = O.down_scale_exp(W, lib=lib)
    cs, ds = O.q4_quantize(W, fp16=True, scale_exp=s, lib=lib)
    ws = O.q4_dequantize(cs, ds, scale_exp=s, lib=lib).astype(np.float64)
    dd = np.repeat(np.abs(ds.astype(np.float64)), 32, axis=1) * 2.0 ** -s
    inner = (cs > 0) & (cs < 15)
    assert np.all(np.abs(ws - W)[inner] <= dd[inner] / 2 * (1 + 1e-6))


ALL_PINS = [pin_exp, pin_topk, pin_topk_golden, pin_csr, pin_csr_golden, pin_placement,
            pin_layer_dense, pin_layer_textbook, pin_layer_special, pin_maxplus, pin_router,
            pin_q4_golden, pin_q4_properties]
