"""Python binding of libestream (the C ABI in include/estream.h).

Argument marshalling only: torch tensors become device/host pointers, the
current torch CUDA stream becomes the ``cuda_stream`` argument, and status
codes become exceptions. Every step of the MoE layer runs in the library's
CUDA kernels; there is no other implementation behind these names, and the
module refuses to load when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libestream.so")

OK, ERR_INVALID_ARG, ERR_CAPACITY, ERR_NOT_BOUND, ERR_CUDA, ERR_PAGER, ERR_TIMEOUT, \
    ERR_DEVICE, ERR_UNSUPPORTED = range(9)
F32, BF16, Q4 = 0, 1, 2
SCHED_AFTER_ROUTING, SCHED_PREFETCH = 0, 1
FFN_AUTO, FFN_SINGLE, FFN_PAIR = 0, 1, 2
PAIR_MIN_ROWS = 160
STATE_NAMES = {0: "Available", 1: "Filling", 2: "Ready", 3: "InUse"}


class EStreamError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)} (status {status})")


class ArenaDesc(ctypes.Structure):
    _fields_ = [
        ("L", ctypes.c_int), ("E", ctypes.c_int), ("H", ctypes.c_int), ("F", ctypes.c_int),
        ("G", ctypes.c_int), ("B", ctypes.c_int), ("Q", ctypes.c_int),
        ("wdtype", ctypes.c_int),
        ("arena_dev", ctypes.c_void_p), ("arena_bytes", ctypes.c_size_t),
        ("host_pool", ctypes.POINTER(ctypes.c_void_p)),
        ("perm", ctypes.POINTER(ctypes.c_int32)),
        ("n_shared", ctypes.c_int), ("F_shared", ctypes.c_int),
        ("shared_dev", ctypes.POINTER(ctypes.c_void_p)),
        ("T_max", ctypes.c_int), ("k_max", ctypes.c_int),
        ("deterministic", ctypes.c_int), ("schedule", ctypes.c_int),
        ("ffn_form", ctypes.c_int),
    ]


class Stats(ctypes.Structure):
    _fields_ = [
        ("calls", ctypes.c_int), ("launches", ctypes.c_int),
        ("ms_route", ctypes.c_double), ("ms_ffn", ctypes.c_double),
        ("ms_shared", ctypes.c_double),
        ("ms_combine", ctypes.c_double), ("ms_total", ctypes.c_double),
        ("n_ffn", ctypes.c_int),
        ("h2d_bytes", ctypes.c_double),
        ("groups_loaded", ctypes.c_int), ("groups_skipped", ctypes.c_int),
        ("groups_hit", ctypes.c_int),
        ("ms_io_busy", ctypes.c_double),
        ("hidden_fraction", ctypes.c_double), ("bubble_rate", ctypes.c_double),
    ]


_lib = None

# name -> (restype, argtypes)
_P, _I, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
SIGNATURES = {
    "estream_status_string": (ctypes.c_char_p, [_I]),
    "estream_version": (_I, []),
    "estream_route_workspace_bytes": (_SZ, [_I, _I, _I, _I]),
    "estream_route_build": (_I, [_P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P, _SZ, _P]),
    "estream_workspace_error": (_I, [_P, _P]),
    "estream_route_build_noalloc": (_I, [_P, _I, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P]),
    "estream_route_noalloc_error": (_I, [_P]),
    "estream_poison_workspace": (_I, [_P, _P]),
    "estream_route_build_from_x": (_I, [_P, _I, _I, _P, _I, _I, _I, _P, _I, _P, _P, _P, _P, _P, _P,
                                        _P, _SZ, _P]),
    "estream_route_build_from_x_fused": (_I, [_I, _I, _I, _I]),
    "estream_moe_layer_prefill_from_x": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P, _P, _P]),
    "estream_router_workspace_bytes": (_SZ, [_I, _I, _I]),
    "estream_router_logits": (_I, [_P, _I, _I, _P, _I, _P, _P, _SZ, _P]),
    "estream_arena_bytes": (_SZ, [_I, _I, _I, _I, _I, _I]),
    "estream_pool_bytes": (_SZ, [_I, _I, _I, _I]),
    "estream_shared_bytes": (_SZ, [_I, _I, _I, _I]),
    "estream_pack_shared": (_I, [ctypes.POINTER(ArenaDesc), _P, _P, _P, _P]),
    "estream_bind_arena": (_I, [ctypes.POINTER(_P), ctypes.POINTER(ArenaDesc)]),
    "estream_pack_experts": (_I, [ctypes.POINTER(ArenaDesc), _I, _P, _P, _P, _P]),
    "estream_arena_preload": (_I, [_P, _I, _P]),
    "estream_arena_invalidate": (_I, [_P]),
    "estream_moe_layer_prefill": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P]),
    "estream_moe_layer_prefill_residual": (_I, [_P, _I, _P, _P, _I, _I, _I, _P, _P, _P]),
    "estream_set_timing": (_I, [_P, _I]),
    "estream_reset_stats": (_I, [_P]),
    "estream_last_stats": (_I, [_P, ctypes.POINTER(Stats)]),
    "estream_get_device_error": (_I, [_P]),
    "estream_residency_trace": (_I, [_P, _P, _I, ctypes.POINTER(_I)]),
    "estream_inject_pager_fault": (_I, [_P, _I, _I]),
    "estream_inject_route_timeout": (_I, [_P]),
    "estream_inject_expert_timeout": (_I, [_P]),
    "estream_pipeline_trace": (_I, [_P, _P, _I, ctypes.POINTER(_I), ctypes.POINTER(ctypes.c_double)]),
    "estream_maxplus_pipeline": (ctypes.c_double, [_P, _P, _I, _I, _I, ctypes.c_double, _P]),
    "estream_bank_bound": (_I, [_I, ctypes.c_double, ctypes.c_double, ctypes.c_double, _I]),
    "estream_autoconfig": (_I, [_I, _P, _P, _P, _P, ctypes.c_double, _I, ctypes.c_double, _P,
                                ctypes.c_double, _I, ctypes.POINTER(_I), ctypes.POINTER(_I),
                                ctypes.POINTER(ctypes.c_double)]),
    "estream_unbind": (None, [_P]),
    "estream_cast_f32_bf16": (_I, [_P, _P, _SZ, _P]),
}


def lib():
    """Load libestream.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libestream.so not found at {LIB_PATH}; build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().estream_status_string(status).decode()


def _check(status: int, where: str) -> None:
    if status != OK:
        raise EStreamError(status, where)


def _dptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream=None, device=None):
    """The cuda_stream argument: `stream` (a torch.cuda.Stream or a raw
    handle), else the current stream of `device`. A torch stream of another
    device than `device` is refused."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    if hasattr(stream, "cuda_stream"):
        if device is not None and stream.device != torch.device(device):
            raise ValueError(f"stream belongs to {stream.device}, the tensors to {device}")
        return stream.cuda_stream
    return stream


class _on(torch.cuda.device):
    """Makes the tensors' device current for the duration of one library
    call: the library launches on the current device, with these pointers."""

    def __init__(self, t: torch.Tensor):
        super().__init__(t.device)


def version() -> int:
    return lib().estream_version()


# ---------------------------------------------------------------------------
# routing + route map
# ---------------------------------------------------------------------------

def route_workspace_bytes(T: int, E: int, k: int, P: int) -> int:
    return lib().estream_route_workspace_bytes(T, E, k, P)


def _need(t: torch.Tensor, numel: int, dtype, name: str, device) -> None:
    """A buffer the library writes or reads through a plain pointer."""
    if t.dtype != dtype or t.numel() < numel or t.device != device:
        raise ValueError(f"{name} must be {dtype} with at least {numel} elements on {device}")


def _check_route_args(logits: torch.Tensor, k: int, phi, P: int, o: dict) -> None:
    if logits.dim() != 2 or logits.dtype != torch.float32 or not logits.is_cuda:
        raise ValueError("logits must be a [T, E] fp32 CUDA tensor")
    T, E = logits.shape
    R = T * k
    dev = logits.device
    if phi is not None:
        _need(phi, E, torch.int32, "phi", dev)
    _need(o["topk_ids"], R, torch.int32, "topk_ids", dev)
    _need(o["alpha"], R, torch.float32, "alpha", dev)
    _need(o["offsets"], P + 2, torch.int32, "offsets", dev)
    _need(o["rec_tok"], R, torch.int32, "rec_tok", dev)
    _need(o["rec_route"], R, torch.int32, "rec_route", dev)


def route_build(logits: torch.Tensor, k: int, renorm: bool, phi: torch.Tensor | None = None,
                P: int | None = None, out: dict | None = None, workspace: torch.Tensor | None = None,
                stream=None) -> dict:
    """estream_route_build on device tensors. Returns a dict with topk_ids,
    alpha, offsets, rec_tok, rec_route (allocated when not given in ``out``)."""
    T, E = logits.shape
    P = E if P is None else P
    dev = logits.device
    R = T * k
    o = dict(out or {})
    o.setdefault("topk_ids", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    o.setdefault("alpha", torch.empty(max(R, 1), dtype=torch.float32, device=dev))
    o.setdefault("offsets", torch.empty(P + 2, dtype=torch.int32, device=dev))
    o.setdefault("rec_tok", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    o.setdefault("rec_route", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    _check_route_args(logits, k, phi, P, o)
    nbytes = route_workspace_bytes(T, E, k, P)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    if workspace.device != dev:
        raise ValueError(f"workspace must be on {dev}")
    with _on(logits):
        st = lib().estream_route_build(
            _dptr(logits), T, E, k, int(bool(renorm)), _dptr(phi), P, _dptr(o["topk_ids"]),
            _dptr(o["alpha"]), _dptr(o["offsets"]), _dptr(o["rec_tok"]), _dptr(o["rec_route"]),
            _dptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream, dev))
    _check(st, "estream_route_build")
    o["workspace"] = workspace
    return o


def router_workspace_bytes(T: int, H: int, E: int) -> int:
    return lib().estream_router_workspace_bytes(T, H, E)


def router_logits(X: torch.Tensor, W_r: torch.Tensor, logits: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """estream_router_logits: logits [T, E] fp32 = X [T, H] bf16 @ W_r [E, H] bf16 ^T."""
    if (X.dim() != 2 or W_r.dim() != 2 or X.dtype != torch.bfloat16 or W_r.dtype != torch.bfloat16
            or W_r.shape[1] != X.shape[1]):
        raise ValueError("X must be [T, H] and W_r [E, H], both bf16")
    if not X.is_cuda or W_r.device != X.device:
        raise ValueError("X and W_r must be on one CUDA device")
    T, H = X.shape
    E = W_r.shape[0]
    if logits is None:
        logits = torch.empty(T, E, dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = torch.empty(max(router_workspace_bytes(T, H, E), 256), dtype=torch.uint8,
                                device=X.device)
    if tuple(logits.shape) != (T, E) or logits.dtype != torch.float32 or logits.device != X.device:
        raise ValueError(f"logits must be [{T}, {E}] fp32 on X's device")
    if workspace.device != X.device:
        raise ValueError("workspace must be on X's device")
    with _on(X):
        st = lib().estream_router_logits(_dptr(X), T, H, _dptr(W_r), E, _dptr(logits),
                                         _dptr(workspace), workspace.numel() * workspace.element_size(),
                                         _stream(stream, X.device))
    _check(st, "estream_router_logits")
    return logits


def route_build_from_x(X: torch.Tensor, W_r: torch.Tensor, k: int, renorm: bool,
                       phi: torch.Tensor | None = None, P: int | None = None, out: dict | None = None,
                       workspace: torch.Tensor | None = None, stream=None) -> dict:
    """estream_route_build_from_x: router logits X W_r^T and the route map in
    one call. Returns route_build's dict plus "logits" [T, E] fp32."""
    if (X.dim() != 2 or W_r.dim() != 2 or X.dtype != torch.bfloat16 or W_r.dtype != torch.bfloat16
            or W_r.shape[1] != X.shape[1]):
        raise ValueError("X must be [T, H] and W_r [E, H], both bf16")
    if not X.is_cuda or W_r.device != X.device:
        raise ValueError("X and W_r must be on one CUDA device")
    T, H = X.shape
    E = W_r.shape[0]
    P = E if P is None else P
    dev = X.device
    R = T * k
    o = dict(out or {})
    o.setdefault("logits", torch.empty(T, E, dtype=torch.float32, device=dev))
    o.setdefault("topk_ids", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    o.setdefault("alpha", torch.empty(max(R, 1), dtype=torch.float32, device=dev))
    o.setdefault("offsets", torch.empty(P + 2, dtype=torch.int32, device=dev))
    o.setdefault("rec_tok", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    o.setdefault("rec_route", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    if tuple(o["logits"].shape) != (T, E) or o["logits"].dtype != torch.float32 \
            or o["logits"].device != dev:
        raise ValueError(f"logits must be [{T}, {E}] fp32 on X's device")
    _check_route_args(o["logits"], k, phi, P, o)
    nbytes = route_workspace_bytes(T, E, k, P)
    if workspace is None:
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
    if workspace.device != dev:
        raise ValueError(f"workspace must be on {dev}")
    with _on(X):
        st = lib().estream_route_build_from_x(
            _dptr(X), T, H, _dptr(W_r), E, k, int(bool(renorm)), _dptr(phi), P, _dptr(o["logits"]),
            _dptr(o["topk_ids"]), _dptr(o["alpha"]), _dptr(o["offsets"]), _dptr(o["rec_tok"]),
            _dptr(o["rec_route"]), _dptr(workspace), workspace.numel() * workspace.element_size(),
            _stream(stream, dev))
    _check(st, "estream_route_build_from_x")
    o["workspace"] = workspace
    return o


def route_build_from_x_fused(T: int, H: int, E: int, P: int | None = None) -> bool:
    """Whether route_build_from_x runs these sizes as one fused launch on
    the current device."""
    return bool(lib().estream_route_build_from_x_fused(T, H, E, E if P is None else P))


def route_build_noalloc(logits: torch.Tensor, k: int, renorm: bool, phi: torch.Tensor | None = None,
                        P: int | None = None, out: dict | None = None, stream=None) -> dict:
    """estream_route_build_noalloc: the same outputs as route_build, with the
    library's static device scratch instead of a caller workspace."""
    T, E = logits.shape
    P = E if P is None else P
    dev = logits.device
    R = T * k
    o = dict(out or {})
    o.setdefault("topk_ids", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    o.setdefault("alpha", torch.empty(max(R, 1), dtype=torch.float32, device=dev))
    o.setdefault("offsets", torch.empty(P + 2, dtype=torch.int32, device=dev))
    o.setdefault("rec_tok", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    o.setdefault("rec_route", torch.empty(max(R, 1), dtype=torch.int32, device=dev))
    _check_route_args(logits, k, phi, P, o)
    with _on(logits):
        st = lib().estream_route_build_noalloc(
            _dptr(logits), T, E, k, int(bool(renorm)), _dptr(phi), P, _dptr(o["topk_ids"]),
            _dptr(o["alpha"]), _dptr(o["offsets"]), _dptr(o["rec_tok"]), _dptr(o["rec_route"]),
            _stream(stream, dev))
    _check(st, "estream_route_build_noalloc")
    return o


def route_noalloc_error(device=None, stream=None) -> int:
    """estream_route_noalloc_error on `device` (default: the current one):
    the status the latest allocation-free route build there recorded."""
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    with torch.cuda.device(device):
        return lib().estream_route_noalloc_error(_stream(stream, device))


def workspace_error(workspace: torch.Tensor, stream=None) -> int:
    with _on(workspace):
        return lib().estream_workspace_error(_dptr(workspace), _stream(stream, workspace.device))


def cast_f32_bf16(src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    if (src.dtype != torch.float32 or dst.dtype != torch.bfloat16 or src.numel() != dst.numel()
            or not src.is_cuda or dst.device != src.device):
        raise ValueError("src must be fp32 and dst bf16 of the same size, on one CUDA device")
    with _on(src):
        _check(lib().estream_cast_f32_bf16(_dptr(src), _dptr(dst), src.numel(),
                                           _stream(stream, src.device)), "estream_cast_f32_bf16")


# ---------------------------------------------------------------------------
# arena / layer
# ---------------------------------------------------------------------------

def arena_bytes(E, H, F, G, B, wdtype) -> int:
    return lib().estream_arena_bytes(E, H, F, G, B, wdtype)


def pool_bytes(E, H, F, wdtype) -> int:
    return lib().estream_pool_bytes(E, H, F, wdtype)


def shared_bytes(n_shared, H, F_shared, wdtype) -> int:
    return lib().estream_shared_bytes(n_shared, H, F_shared, wdtype)


def pack_shared(desc: ArenaDesc, sg: torch.Tensor, su: torch.Tensor, sd: torch.Tensor,
                out: torch.Tensor) -> None:
    for t in (sg, su, sd, out):
        assert t.device.type == "cpu" and t.is_contiguous()
    _check(lib().estream_pack_shared(ctypes.byref(desc), sg.data_ptr(), su.data_ptr(),
                                     sd.data_ptr(), out.data_ptr()), "estream_pack_shared")


def make_desc(L, E, H, F, G, B, wdtype, arena: torch.Tensor, pools, perm=None, n_shared=0,
              F_shared=0, shared=None, T_max=1, k_max=1, deterministic=False,
              schedule=SCHED_AFTER_ROUTING, Q=1, ffn_form=FFN_AUTO):
    """Fill an ArenaDesc; returns (desc, keepalive) -- keep both alive while bound."""
    d = ArenaDesc()
    d.L, d.E, d.H, d.F, d.G, d.B, d.Q = L, E, H, F, G, B, Q
    d.wdtype = wdtype
    d.arena_dev = arena.data_ptr() if arena is not None else None
    d.arena_bytes = arena.numel() * arena.element_size() if arena is not None else 0
    pool_arr = (ctypes.c_void_p * L)(*[p.data_ptr() if p is not None else None for p in pools])
    d.host_pool = ctypes.cast(pool_arr, ctypes.POINTER(ctypes.c_void_p))
    keep = [pool_arr]
    if perm is not None:
        perm_arr = (ctypes.c_int32 * (L * E))(*[int(v) for v in torch.as_tensor(perm).reshape(-1).tolist()])
        d.perm = ctypes.cast(perm_arr, ctypes.POINTER(ctypes.c_int32))
        keep.append(perm_arr)
    d.n_shared, d.F_shared = n_shared, F_shared
    if n_shared and shared is not None:
        sh_arr = (ctypes.c_void_p * L)(*[s.data_ptr() for s in shared])
        d.shared_dev = ctypes.cast(sh_arr, ctypes.POINTER(ctypes.c_void_p))
        keep.append(sh_arr)
    d.T_max, d.k_max = T_max, k_max
    d.deterministic = int(bool(deterministic))
    d.schedule = schedule
    d.ffn_form = ffn_form
    return d, keep


def pack_experts(desc: ArenaDesc, layer: int, wg: torch.Tensor, wu: torch.Tensor, wd: torch.Tensor,
                 pool_out: torch.Tensor) -> None:
    for t in (wg, wu, wd, pool_out):
        assert t.device.type == "cpu" and t.is_contiguous()
    _check(lib().estream_pack_experts(ctypes.byref(desc), layer, wg.data_ptr(), wu.data_ptr(),
                                      wd.data_ptr(), pool_out.data_ptr()), "estream_pack_experts")


def bind_arena(desc: ArenaDesc) -> int:
    ctx = ctypes.c_void_p()
    _check(lib().estream_bind_arena(ctypes.byref(ctx), ctypes.byref(desc)), "estream_bind_arena")
    return ctx.value


def arena_preload(ctx, layer: int, stream=None) -> None:
    _check(lib().estream_arena_preload(ctx, layer, _stream(stream)), "estream_arena_preload")


def arena_invalidate(ctx) -> None:
    _check(lib().estream_arena_invalidate(ctx), "estream_arena_invalidate")


def _check_layer_args(X: torch.Tensor, logits: torch.Tensor | None, Y: torch.Tensor,
                      A: torch.Tensor | None = None) -> None:
    """Shapes and types the layer call reads and writes through plain
    pointers: X [T, H] (bf16 or fp32), logits [T, E] fp32 (when given), Y
    [T, H] fp32 and the residual A like X, all on one CUDA device."""
    if X.dim() != 2 or Y.dim() != 2 or (logits is not None and logits.dim() != 2):
        raise ValueError("X, logits and Y must be 2-d")
    T, H = X.shape
    if (logits is not None and logits.shape[0] != T) or tuple(Y.shape) != (T, H):
        raise ValueError(f"logits must be [T, E] and Y [T, H] with T={T}, H={H}")
    if X.dtype not in (torch.bfloat16, torch.float32):
        raise ValueError("X must be bf16 or fp32")
    if (logits is not None and logits.dtype != torch.float32) or Y.dtype != torch.float32:
        raise ValueError("logits and Y must be fp32")
    if A is not None and (tuple(A.shape) != (T, H) or A.dtype != X.dtype):
        raise ValueError("the residual must have X's shape and type")
    tensors = [X, Y] + [t for t in (logits, A) if t is not None]
    if any(not t.is_cuda for t in tensors) or len({t.device for t in tensors}) != 1:
        raise ValueError("X, logits, Y (and the residual) must be on one CUDA device")


def moe_layer_prefill(ctx, layer: int, X: torch.Tensor, logits: torch.Tensor, k: int,
                      renorm: bool, Y: torch.Tensor, stream=None) -> None:
    _check_layer_args(X, logits, Y)
    T = X.shape[0]
    with _on(X):
        _check(lib().estream_moe_layer_prefill(ctx, layer, _dptr(X), _dptr(logits), T, k,
                                               int(bool(renorm)), _dptr(Y), _stream(stream, X.device)),
               "estream_moe_layer_prefill")


def moe_layer_prefill_residual(ctx, layer: int, X: torch.Tensor, logits: torch.Tensor, k: int,
                               renorm: bool, A: torch.Tensor, Y: torch.Tensor, stream=None) -> None:
    """Y = A + the layer's MoE output (Y written, not read)."""
    _check_layer_args(X, logits, Y, A)
    T = X.shape[0]
    with _on(X):
        _check(lib().estream_moe_layer_prefill_residual(ctx, layer, _dptr(X), _dptr(logits), T, k,
                                                        int(bool(renorm)), _dptr(A), _dptr(Y),
                                                        _stream(stream, X.device)),
               "estream_moe_layer_prefill_residual")


def moe_layer_prefill_from_x(ctx, layer: int, X: torch.Tensor, W_r: torch.Tensor, k: int,
                             renorm: bool, Y: torch.Tensor, A: torch.Tensor | None = None,
                             logits_out: torch.Tensor | None = None, stream=None) -> None:
    """Routing from the layer input (router logits, top-k and route map in
    one launch), then the experts: Y += MoE(X), or Y = A + MoE(X)."""
    if W_r.dim() != 2 or W_r.dtype != torch.bfloat16 or W_r.shape[1] != X.shape[1] \
            or W_r.device != X.device:
        raise ValueError("W_r must be [E, H] bf16 on X's device")
    T = X.shape[0]
    E = W_r.shape[0]
    if logits_out is not None and tuple(logits_out.shape) != (T, E):
        raise ValueError(f"logits_out must be [{T}, {E}]")
    _check_layer_args(X, logits_out, Y, A)
    with _on(X):
        _check(lib().estream_moe_layer_prefill_from_x(ctx, layer, _dptr(X), _dptr(W_r), T, k,
                                                      int(bool(renorm)), _dptr(A), _dptr(Y),
                                                      _dptr(logits_out), _stream(stream, X.device)),
               "estream_moe_layer_prefill_from_x")


def set_timing(ctx, on: bool) -> None:
    _check(lib().estream_set_timing(ctx, int(bool(on))), "estream_set_timing")


def reset_stats(ctx) -> None:
    _check(lib().estream_reset_stats(ctx), "estream_reset_stats")


def last_stats(ctx) -> dict:
    s = Stats()
    _check(lib().estream_last_stats(ctx, ctypes.byref(s)), "estream_last_stats")
    return {name: getattr(s, name) for name, _ in Stats._fields_}


def get_device_error(ctx) -> int:
    return lib().estream_get_device_error(ctx)


def poison_workspace(ctx, stream=None) -> None:
    """estream_poison_workspace (test aid): NaN / past-target fill of the
    context's per-call buffers on the stream, before a layer call."""
    _check(lib().estream_poison_workspace(ctx, _stream(stream)), "estream_poison_workspace")


def residency_trace(ctx, cap: int = 4096):
    buf = (ctypes.c_int32 * (4 * cap))()
    n = ctypes.c_int()
    _check(lib().estream_residency_trace(ctx, buf, cap, ctypes.byref(n)), "estream_residency_trace")
    m = min(n.value, cap)
    return [tuple(buf[4 * i:4 * i + 4]) for i in range(m)]


def pipeline_trace(ctx, cap: int = 4096):
    """Per-group (a, d, s, f) times in ms of the last timed paged call, and
    the time routing finished."""
    import numpy as np
    buf = np.zeros((cap, 4), dtype=np.float64)
    n = ctypes.c_int()
    tne = ctypes.c_double()
    _check(lib().estream_pipeline_trace(ctx, buf.ctypes.data_as(ctypes.c_void_p), cap,
                                        ctypes.byref(n), ctypes.byref(tne)), "estream_pipeline_trace")
    return buf[:min(n.value, cap)].copy(), tne.value


def maxplus_pipeline(L, X, q: int, b: int, T_ne: float = 0.0):
    """Eq. 5: returns (T_pipe, adsf[K][4])."""
    import numpy as np
    L = np.ascontiguousarray(L, dtype=np.float64)
    X = np.ascontiguousarray(X, dtype=np.float64)
    K = len(L)
    out = np.zeros((max(K, 1), 4), dtype=np.float64)
    t = lib().estream_maxplus_pipeline(L.ctypes.data_as(ctypes.c_void_p), X.ctypes.data_as(ctypes.c_void_p),
                                       K, q, b, T_ne, out.ctypes.data_as(ctypes.c_void_p))
    return t, out[:K]


def bank_bound(g, M_max, M_other, W_e, N_e) -> int:
    return lib().estream_bank_bound(g, M_max, M_other, W_e, N_e)


def autoconfig(profiles: dict, T_ne: float, Q0: int, M_max: float, W_e: float, N_e: int,
               M_other: dict | None = None):
    """Eqs. 9-10 over {g: (L[], X[])}. Returns (G*, B*, T_pipe*)."""
    import numpy as np
    gs = list(profiles)
    Ls = [np.ascontiguousarray(profiles[g][0], dtype=np.float64) for g in gs]
    Xs = [np.ascontiguousarray(profiles[g][1], dtype=np.float64) for g in gs]
    g_arr = (ctypes.c_int * len(gs))(*gs)
    k_arr = (ctypes.c_int * len(gs))(*[len(x) for x in Ls])
    L_arr = (ctypes.c_void_p * len(gs))(*[x.ctypes.data for x in Ls])
    X_arr = (ctypes.c_void_p * len(gs))(*[x.ctypes.data for x in Xs])
    mo = None
    if M_other is not None:
        mo = (ctypes.c_double * len(gs))(*[float(M_other[g]) for g in gs])
    G, B, T = ctypes.c_int(), ctypes.c_int(), ctypes.c_double()
    _check(lib().estream_autoconfig(len(gs), g_arr, k_arr, L_arr, X_arr, T_ne, Q0, M_max, mo, W_e,
                                    N_e, ctypes.byref(G), ctypes.byref(B), ctypes.byref(T)),
           "estream_autoconfig")
    return G.value, B.value, T.value


def inject_expert_timeout(ctx) -> None:
    _check(lib().estream_inject_expert_timeout(ctx), "estream_inject_expert_timeout")


def inject_route_timeout(ctx) -> None:
    _check(lib().estream_inject_route_timeout(ctx), "estream_inject_route_timeout")


def inject_pager_fault(ctx, layer: int, group: int) -> None:
    _check(lib().estream_inject_pager_fault(ctx, layer, group), "estream_inject_pager_fault")


def unbind(ctx) -> None:
    if ctx:
        lib().estream_unbind(ctx)
