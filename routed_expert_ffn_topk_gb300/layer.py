"""Owner of the memory one bound arena needs, for a Workload.

Allocates (through torch) the device arena, the pinned host pools packed by
``estream_pack_experts``, the packed shared experts on the device, and binds
the library context. ``prefill`` is the C-ABI layer call. Nothing here
computes any part of the layer.
"""
from __future__ import annotations

import torch

from . import estream as es
from .workloads import Workload, ceil_div


class BoundLayerStack:
    """One arena bound for every layer of a workload.

    mode="resident": B = ceil(E/G) banks and every layer's groups preloaded
    (only for single-layer workloads); mode="paged": the workload's (G, B).
    """

    def __init__(self, wl: Workload, mode: str = "resident", perm=None, G=None, B=None,
                 deterministic=False, schedule=es.SCHED_AFTER_ROUTING, T_max=None, k_max=None,
                 Q=1, ffn_form=es.FFN_AUTO, wdtype=None, device="cuda"):
        cfg = wl.cfg
        self.cfg, self.wl, self.mode = cfg, wl, mode
        device = torch.device(device)
        if device.type == "cuda" and device.index is None:
            device = torch.device("cuda", torch.cuda.current_device())
        self.device = device
        # wdtype=es.Q4 packs the (bf16) weights of a bf16 workload as 4-bit experts
        self.dtype = wdtype if wdtype is not None else (es.BF16 if cfg.dtype == "bf16" else es.F32)
        L = len(wl.layers)
        G = G or cfg.G
        if mode == "resident":
            B = B or ceil_div(cfg.E, G)
        else:
            B = B or cfg.B
        self.G, self.B = G, B
        self.T_max = T_max or cfg.T
        self.k_max = k_max or cfg.k
        if perm is None:
            perm = torch.arange(cfg.E, dtype=torch.int32).repeat(L, 1)
        self.perm = torch.as_tensor(perm, dtype=torch.int32).reshape(L, cfg.E)
        self.arena = torch.empty(es.arena_bytes(cfg.E, cfg.H, cfg.F, G, B, self.dtype),
                                 dtype=torch.uint8, device=device)
        pin = torch.cuda.is_available()
        nbytes = es.pool_bytes(cfg.E, cfg.H, cfg.F, self.dtype)
        self.pools = [torch.empty(nbytes, dtype=torch.uint8, pin_memory=pin) for _ in range(L)]
        self.shared = []
        desc, keep = es.make_desc(L, cfg.E, cfg.H, cfg.F, G, B, self.dtype, self.arena, self.pools,
                                  perm=self.perm, n_shared=cfg.n_shared, F_shared=cfg.F_shared,
                                  shared=None, T_max=self.T_max, k_max=self.k_max,
                                  deterministic=deterministic, schedule=schedule)
        for l, lw in enumerate(wl.layers):
            es.pack_experts(desc, l, lw.Wg.contiguous(), lw.Wu.contiguous(), lw.Wd.contiguous(),
                            self.pools[l])
            if cfg.n_shared:
                buf = torch.empty(es.shared_bytes(cfg.n_shared, cfg.H, cfg.F_shared, self.dtype),
                                  dtype=torch.uint8)
                es.pack_shared(desc, lw.Sg.contiguous(), lw.Su.contiguous(), lw.Sd.contiguous(), buf)
                self.shared.append(buf.to(device))
        self.desc, self.keep = es.make_desc(
            L, cfg.E, cfg.H, cfg.F, G, B, self.dtype, self.arena, self.pools, perm=self.perm,
            n_shared=cfg.n_shared, F_shared=cfg.F_shared, shared=self.shared or None,
            T_max=self.T_max, k_max=self.k_max, deterministic=deterministic, schedule=schedule, Q=Q,
            ffn_form=ffn_form)
        if mode == "resident" and L != 1:
            raise ValueError("resident mode holds one layer")
        # the context lives on the arena's device: bind and preload with it current
        with torch.cuda.device(device):
            self.ctx = es.bind_arena(self.desc)
            if mode == "resident":
                es.arena_preload(self.ctx, 0)

    def prefill(self, layer: int, X: torch.Tensor, logits: torch.Tensor, Y: torch.Tensor,
                k=None, renorm=None, stream=None, residual: torch.Tensor | None = None) -> None:
        """Y += MoE(X), or Y = residual + MoE(X) when `residual` is given."""
        cfg = self.cfg
        if X.dim() != 2 or X.shape[1] != cfg.H or logits.dim() != 2 or logits.shape[1] != cfg.E:
            raise ValueError(f"X must be [T, {cfg.H}] and logits [T, {cfg.E}]")
        want = torch.float32 if self.dtype == es.F32 else torch.bfloat16
        if X.dtype != want:
            raise ValueError(f"X must be {want} for this arena")
        if X.device != self.device:
            raise ValueError(f"X is on {X.device}, the arena on {self.device}")
        k = cfg.k if k is None else k
        renorm = cfg.renorm if renorm is None else renorm
        if residual is None:
            es.moe_layer_prefill(self.ctx, layer, X, logits, k, renorm, Y, stream)
        else:
            es.moe_layer_prefill_residual(self.ctx, layer, X, logits, k, renorm, residual, Y, stream)

    def prefill_from_router(self, layer: int, X: torch.Tensor, W_r: torch.Tensor, Y: torch.Tensor,
                            k=None, renorm=None, stream=None) -> torch.Tensor:
        """Router logits = X W_r^T (estream_router_logits), then the layer call;
        returns the logits (kept in a buffer reused across calls)."""
        T = X.shape[0]
        E = W_r.shape[0]
        buf = getattr(self, "_router_buf", None)
        if buf is None or buf[0].shape[0] < T * E or buf[1].device != X.device:
            ws_bytes = max(es.router_workspace_bytes(self.T_max, X.shape[1], E), 256)
            buf = (torch.empty(self.T_max * E, dtype=torch.float32, device=X.device),
                   torch.empty(ws_bytes, dtype=torch.uint8, device=X.device))
            self._router_buf = buf
        logits = buf[0][:T * E].view(T, E)
        es.router_logits(X, W_r, logits=logits, workspace=buf[1], stream=stream)
        self.prefill(layer, X, logits, Y, k=k, renorm=renorm, stream=stream)
        return logits

    def poison(self, stream=None) -> None:
        """Test aid: NaN / past-target fill of the context's per-call buffers
        (estream_poison_workspace) on the stream, before a layer call."""
        with torch.cuda.device(self.device):
            es.poison_workspace(self.ctx, stream)

    def prefill_from_x(self, layer: int, X: torch.Tensor, W_r: torch.Tensor, Y: torch.Tensor,
                       k=None, renorm=None, stream=None, residual: torch.Tensor | None = None,
                       logits_out: torch.Tensor | None = None) -> None:
        """The layer call with routing from X and the router weights W_r [E, H]
        (estream_moe_layer_prefill_from_x): Y += MoE(X), or Y = residual +
        MoE(X); the router logits go to logits_out when given."""
        cfg = self.cfg
        if X.dim() != 2 or X.shape[1] != cfg.H or X.dtype != torch.bfloat16 or X.device != self.device:
            raise ValueError(f"X must be [T, {cfg.H}] bf16 on {self.device}")
        if W_r.shape[0] != cfg.E:
            raise ValueError(f"W_r must have {cfg.E} rows")
        k = cfg.k if k is None else k
        renorm = cfg.renorm if renorm is None else renorm
        es.moe_layer_prefill_from_x(self.ctx, layer, X, W_r, k, renorm, Y, A=residual,
                                    logits_out=logits_out, stream=stream)

    def close(self) -> None:
        if getattr(self, "ctx", None):
            with torch.cuda.device(self.device):
                es.unbind(self.ctx)
            self.ctx = None

    def __del__(self):  # pragma: no cover
        try:
            self.close()
        except Exception:
            pass
