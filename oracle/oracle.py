"""Python face of the CPU oracle (``estream_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
bench's CPU-baseline leg import this module. The product library never calls
it and shares no code with it.

Every function states the passage of "EStream: Fast and Memory-Efficient MoE
Prefill through Expert Virtualization on Mobile NPUs" it restates; the C file
holds the arithmetic. ``build()`` compiles the C file with gcc (plain -O2, no
fast-math, ``-ffp-contract=off`` so every written rounding step is kept).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "estream_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def _compile(src: str, out: str, extra_flags=()) -> None:
    os.makedirs(os.path.dirname(out), exist_ok=True)
    base = ["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared"]
    tmp = out + ".tmp%d" % os.getpid()
    try:
        subprocess.run(base + ["-fopenmp"] + list(extra_flags) + [src, "-o", tmp, "-lm"],
                       check=True, capture_output=True)
    except subprocess.CalledProcessError:
        # no OpenMP runtime: the oracle runs on one thread
        subprocess.run(base + list(extra_flags) + [src, "-o", tmp, "-lm"],
                       check=True, capture_output=True)
    os.replace(tmp, out)


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (if stale)."""
    if force or not os.path.exists(_LIB_PATH) or \
            os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        _compile(_SRC, _LIB_PATH)
    return _LIB_PATH


def _declare(lib) -> None:
    P = ctypes.c_void_p
    i = ctypes.c_int
    lib.oracle_exp_f32.argtypes = [ctypes.c_float]
    lib.oracle_exp_f32.restype = ctypes.c_float
    lib.oracle_route_topk.argtypes = [P, i, i, i, i, P, P]
    lib.oracle_route_topk.restype = i
    lib.oracle_route_csr.argtypes = [P, i, i, P, i, i, P, P, P]
    lib.oracle_route_csr.restype = i
    lib.oracle_grouped_placement.argtypes = [P, i, i, P, P]
    lib.oracle_grouped_placement.restype = i
    lib.oracle_moe_layer_rows.argtypes = [P, i, i, i, i, i, P, P, P, P, P,
                                          i, i, P, P, P, P, i, P, i, P]
    lib.oracle_moe_layer_rows.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    lib.oracle_maxplus.argtypes = [P, P, i, i, i, ctypes.c_double, P]
    lib.oracle_maxplus.restype = ctypes.c_double
    lib.oracle_router_logits.argtypes = [P, i, i, P, i, i, P]
    lib.oracle_router_logits.restype = i
    lib.oracle_down_scale_exp.argtypes = [P, ctypes.c_size_t, i]
    lib.oracle_down_scale_exp.restype = i
    lib.oracle_q4_quantize.argtypes = [P, i, i, i, i, i, P, P]
    lib.oracle_q4_quantize.restype = i
    lib.oracle_q4_dequantize.argtypes = [P, P, i, i, i, P]
    lib.oracle_q4_dequantize.restype = i


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` selects
    another build of the same source (the tests use this for planted
    mistakes)."""
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
        _declare(lib)
        return lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            _declare(lib)
            _lib = lib
    return _lib


def _ptr(a: np.ndarray | None):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _as_weight(a):
    """fp32 arrays pass as fp32; bf16 data passes as its uint16 bit pattern.
    Accepts numpy arrays or torch tensors (bf16 tensors are viewed as int16)."""
    try:
        import torch
        if isinstance(a, torch.Tensor):
            a = a.detach().cpu().contiguous()
            if a.dtype == torch.bfloat16:
                return np.ascontiguousarray(a.view(torch.int16).numpy().view(np.uint16)), 1
            return np.ascontiguousarray(a.to(torch.float32).numpy()), 0
    except ImportError:  # pragma: no cover
        pass
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        return a, 1
    return np.ascontiguousarray(a, dtype=np.float32), 0


def exp_f32(x, lib=None) -> np.ndarray:
    """The written fp32 exponential (Cody & Waite reduction + degree-7 Taylor)."""
    lib = lib or load()
    x = np.asarray(x, dtype=np.float32).ravel()
    return np.array([lib.oracle_exp_f32(float(v)) for v in x], dtype=np.float32)


def route_topk(logits, k: int, renorm: bool, lib=None):
    """Softmax top-k router: (topk_ids [T,k] int32, alpha [T,k] fp32).

    The pages say a router assigns each token to the top-k of E experts
    (section 2.2) and that routes carry (e_i, t_i, alpha_i) (section 3.2);
    score function, renormalisation and tie-break are the readings stated in
    the C file."""
    lib = lib or load()
    lg = np.ascontiguousarray(logits, dtype=np.float32)
    T, E = lg.shape
    ids = np.zeros((T, k), dtype=np.int32)
    alpha = np.zeros((T, k), dtype=np.float32)
    rc = lib.oracle_route_topk(_ptr(lg), T, E, k, int(bool(renorm)), _ptr(ids), _ptr(alpha))
    if rc != 0:
        raise ValueError("oracle_route_topk: bad arguments")
    return ids, alpha


def route_csr(topk_ids, E: int, P: int, phi=None, lib=None):
    """Route map of section 3.2 / Algorithm 1: (offsets [P+2], rec_tok [R],
    rec_route [R]); slot P collects routes whose expert is not resident."""
    lib = lib or load()
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, k = ids.shape
    R = T * k
    offsets = np.zeros(P + 2, dtype=np.int32)
    rec_tok = np.zeros(max(R, 1), dtype=np.int32)
    rec_route = np.zeros(max(R, 1), dtype=np.int32)
    ph = None if phi is None else np.ascontiguousarray(phi, dtype=np.int32)
    rc = lib.oracle_route_csr(_ptr(ids), T, k, _ptr(ph), E, P, _ptr(offsets),
                              _ptr(rec_tok), _ptr(rec_route))
    if rc != 0:
        raise ValueError("oracle_route_csr: bad arguments")
    return offsets, rec_tok[:R], rec_route[:R]


def grouped_placement(perm, E: int, G: int, bank_of_group, lib=None) -> np.ndarray:
    """Eq. 4: phi[e] = b*G + (pi(e) mod G) for group floor(pi(e)/G) in bank b."""
    lib = lib or load()
    pm = None if perm is None else np.ascontiguousarray(perm, dtype=np.int32)
    bq = np.ascontiguousarray(bank_of_group, dtype=np.int32)
    phi = np.zeros(E, dtype=np.int32)
    if lib.oracle_grouped_placement(_ptr(pm), E, G, _ptr(bq), _ptr(phi)) != 0:
        raise ValueError("oracle_grouped_placement: bad arguments")
    return phi


def moe_layer_rows(X, Wg, Wu, Wd, topk_ids, alpha, rows=None, shared=None,
                   residual=None, lib=None) -> np.ndarray:
    """Eq. 2 with Eq. 1, in fp64, for the token rows listed in ``rows``
    (all tokens when None). Returns Y[len(rows), H] (float64).

    X [T,H]; Wg, Wu [E,F,H]; Wd [E,H,F]; shared = (Sg [S,Fs,H], Su, Sd [S,H,Fs])
    with weight 1 each; residual = A [T,H] or None (zero)."""
    lib = lib or load()
    Xa, bx = _as_weight(X)
    ga, bg = _as_weight(Wg)
    ua, bu = _as_weight(Wu)
    da, bd = _as_weight(Wd)
    if not (bx == bg == bu == bd):
        raise ValueError("X and the weights must share one encoding")
    T, H = Xa.shape
    E, F, H2 = ga.shape
    assert H2 == H and ua.shape == ga.shape and da.shape == (E, H, F)
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32).reshape(T, -1)
    al = np.ascontiguousarray(alpha, dtype=np.float32).reshape(T, -1)
    k = ids.shape[1]
    r = np.arange(T, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    n_shared, Fs, sg, su, sd = 0, 0, None, None, None
    if shared is not None:
        sg, bsg = _as_weight(shared[0])
        su, bsu = _as_weight(shared[1])
        sd, bsd = _as_weight(shared[2])
        if not (bsg == bsu == bsd == bx):
            raise ValueError("shared weights must share X's encoding")
        n_shared, Fs = sg.shape[0], sg.shape[1]
    A = None if residual is None else np.ascontiguousarray(residual, dtype=np.float64)
    Y = np.zeros((len(r), H), dtype=np.float64)
    rc = lib.oracle_moe_layer_rows(_ptr(Xa), T, H, E, F, k, _ptr(ga), _ptr(ua), _ptr(da),
                                   _ptr(ids), _ptr(al), n_shared, Fs, _ptr(sg), _ptr(su),
                                   _ptr(sd), _ptr(A), bx, _ptr(r), len(r), _ptr(Y))
    if rc != 0:
        raise ValueError("oracle_moe_layer_rows: bad arguments")
    return Y


def maxplus(L, X, q: int, b: int, T_ne: float = 0.0, lib=None):
    """Section 3.4, Eq. 5: (T_pipe, per-group (a, d, s, f))."""
    lib = lib or load()
    L = np.ascontiguousarray(L, dtype=np.float64)
    X = np.ascontiguousarray(X, dtype=np.float64)
    K = len(L)
    out = np.zeros((max(K, 1), 4), dtype=np.float64)
    t = lib.oracle_maxplus(_ptr(L), _ptr(X), K, q, b, float(T_ne), _ptr(out))
    return t, out[:K]


def router_logits(X, W_r, lib=None) -> np.ndarray:
    """Router logits l[t][e] = sum_h X[t][h] * W_r[e][h] in fp64 (the linear
    router upstream of the top-k; reading stated in the C file)."""
    lib = lib or load()
    Xa, bx = _as_weight(X)
    Wa, bw = _as_weight(W_r)
    if bx != bw:
        raise ValueError("X and W_r must share one encoding")
    T, H = Xa.shape
    E, H2 = Wa.shape
    if H2 != H:
        raise ValueError("X and W_r disagree on H")
    out = np.zeros((T, E), dtype=np.float64)
    if lib.oracle_router_logits(_ptr(Xa), T, H, _ptr(Wa), E, bx, _ptr(out)) != 0:
        raise ValueError("oracle_router_logits: bad arguments")
    return out


def down_scale_exp(W, lib=None) -> int:
    """The power-of-two exponent s applied to a down plane before it is
    quantised or converted (its largest magnitude lands in [2^14, 2^15))."""
    lib = lib or load()
    a, b = _as_weight(W)
    return lib.oracle_down_scale_exp(_ptr(a), a.size, b)


def q4_quantize(W, fp16: bool, scale_exp: int = 0, lib=None):
    """Q4_0-style block quantisation of a [rows][cols] matrix along cols:
    (codes [rows][cols] uint8 in 0..15, d [rows][cols/32] fp32)."""
    lib = lib or load()
    a, b = _as_weight(W)
    rows, cols = a.shape
    codes = np.zeros((rows, cols), dtype=np.uint8)
    d = np.zeros((rows, cols // 32), dtype=np.float32)
    if lib.oracle_q4_quantize(_ptr(a), rows, cols, b, scale_exp, int(bool(fp16)), _ptr(codes),
                              _ptr(d)) != 0:
        raise ValueError("oracle_q4_quantize: bad arguments")
    return codes, d


def q4_dequantize(codes, d, scale_exp: int = 0, lib=None) -> np.ndarray:
    """w = (q - 8) * d * 2^-scale_exp as fp32."""
    lib = lib or load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    d = np.ascontiguousarray(d, dtype=np.float32)
    rows, cols = codes.shape
    w = np.zeros((rows, cols), dtype=np.float32)
    if lib.oracle_q4_dequantize(_ptr(codes), _ptr(d), rows, cols, scale_exp, _ptr(w)) != 0:
        raise ValueError("oracle_q4_dequantize: bad arguments")
    return w


def num_threads(lib=None) -> int:
    return (lib or load()).oracle_num_threads()
