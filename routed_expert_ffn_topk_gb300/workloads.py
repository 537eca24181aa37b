"""Seeded synthetic workloads for one MoE layer's prefill.

This module only draws random inputs; it holds none of the method's
arithmetic (no softmax, no top-k, no FFN), so both the CUDA path and the CPU
oracle can consume what it makes.

Five layer shapes are provided, named for the model family whose dimensions
they copy. Every tensor comes from a ``torch.Generator`` (CPU) seeded with
``1000 + config number``, drawn in a fixed order: router logits, per-expert
logit bias, activations X, then per layer and per expert W_g, W_u, W_d, then
the shared experts. bf16 values are torch's round-to-nearest-even of the
fp32 draw.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class LayerConfig:
    key: str
    name: str
    T: int            # prompt tokens
    H: int            # hidden size
    E: int            # routed experts
    k: int            # experts per token
    F: int            # routed expert FFN size
    dtype: str        # "bf16" or "f32" for X and weights
    renorm: bool      # renormalise the selected softmax weights
    P: int            # arena slots when paged (= B * G)
    G: int            # experts per storage group / bank
    B: int            # banks
    n_shared: int = 0  # always-on shared experts (weight 1)
    F_shared: int = 0
    layers: int = 1
    logits: str = "normal"   # "normal", "normal+bias", "zipf-gumbel"
    x_std: float = 1.0
    w_std: float = 0.02
    bias_std: float = 0.5
    zipf_s: float = 1.1

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def elem_bytes(self) -> int:
        return 2 if self.dtype == "bf16" else 4

    def expert_bytes(self) -> int:
        """Packed size W_e of one routed expert (gate, up and down planes)."""
        return 3 * self.H * self.F * self.elem_bytes

    def flops_per_layer(self) -> float:
        """Algorithmic FLOPs: 2 flops per multiply-add over the three
        projections of every route, plus the shared experts over every token."""
        return 6.0 * self.H * self.F * self.T * self.k + \
            6.0 * self.H * self.F_shared * self.T * self.n_shared


CONFIGS = {
    "c1": LayerConfig("c1", "tiny MoE layer", T=64, H=256, E=8, k=2, F=512, dtype="f32",
                      renorm=False, P=8, G=8, B=1, x_std=0.02),
    "c2": LayerConfig("c2", "OLMoE-shaped layer", T=1024, H=2048, E=64, k=8, F=1024,
                      dtype="bf16", renorm=False, P=16, G=8, B=2, logits="normal+bias"),
    "c3": LayerConfig("c3", "DeepSeek-V2-Lite-shaped layer", T=2048, H=2048, E=64, k=6,
                      F=1408, dtype="bf16", renorm=True, P=24, G=8, B=3, n_shared=2,
                      F_shared=1408),
    "c4": LayerConfig("c4", "Qwen-MoE-shaped layer stack", T=4096, H=2048, E=60, k=4,
                      F=1408, dtype="bf16", renorm=False, P=16, G=8, B=2, n_shared=1,
                      F_shared=5632, layers=4, logits="zipf-gumbel"),
    "c5": LayerConfig("c5", "Mixtral-shaped layer", T=4096, H=4096, E=8, k=2, F=14336,
                      dtype="bf16", renorm=True, P=2, G=1, B=2),
}
CONFIG_SEEDS = {"c1": 1001, "c2": 1002, "c3": 1003, "c4": 1004, "c5": 1005}


def scaled(cfg: LayerConfig, T=None, H=None, E=None, k=None, F=None, F_shared=None,
           layers=None, key_suffix="-small") -> LayerConfig:
    """The same family with smaller sizes (for oracle-sized parity runs)."""
    kw = {}
    for name, v in (("T", T), ("H", H), ("E", E), ("k", k), ("F", F),
                    ("F_shared", F_shared), ("layers", layers)):
        if v is not None:
            kw[name] = v
    out = dataclasses.replace(cfg, key=cfg.key + key_suffix, **kw)
    E2 = out.E
    P = min(out.P, E2)
    G = min(out.G, P)
    B = max(1, P // G)
    return dataclasses.replace(out, P=B * G, G=G, B=B)


@dataclasses.dataclass
class LayerWeights:
    Wg: torch.Tensor          # [E, F, H]
    Wu: torch.Tensor          # [E, F, H]
    Wd: torch.Tensor          # [E, H, F]
    Sg: torch.Tensor | None   # [n_shared, Fs, H]
    Su: torch.Tensor | None
    Sd: torch.Tensor | None   # [n_shared, H, Fs]


@dataclasses.dataclass
class Workload:
    cfg: LayerConfig
    logits: list              # per layer [T, E] fp32
    X: torch.Tensor           # [T, H] (first layer's input)
    layers: list              # per layer LayerWeights


def make_router(T: int, H: int, E: int, seed: int, dtype=torch.bfloat16):
    """Seeded inputs of the router upstream of the top-k, drawn from their own
    generator (so the layer workloads' draws are unchanged): X [T, H] ~ N(0, 1)
    and W_r [E, H] ~ N(0, 1/H), giving logits of about unit variance."""
    gen = torch.Generator().manual_seed(seed)
    X = torch.randn((T, H), generator=gen, dtype=torch.float32).to(dtype)
    W_r = (torch.randn((E, H), generator=gen, dtype=torch.float32) / math.sqrt(H)).to(dtype)
    return X, W_r


def _randn(gen, shape, std, dtype):
    return (torch.randn(shape, generator=gen, dtype=torch.float32) * std).to(dtype)


def _logits(cfg: LayerConfig, gen) -> torch.Tensor:
    T, E = cfg.T, cfg.E
    if cfg.logits == "normal":
        return torch.randn((T, E), generator=gen, dtype=torch.float32)
    if cfg.logits == "normal+bias":
        base = torch.randn((T, E), generator=gen, dtype=torch.float32)
        bias = torch.randn((E,), generator=gen, dtype=torch.float32) * cfg.bias_std
        return base + bias[None, :]
    if cfg.logits == "zipf-gumbel":
        # Gumbel-top-k sampling: the k largest of log p_e + Gumbel(0,1) are k
        # draws without replacement from p (Vieira 2014; Kool et al. 2019),
        # with p_e proportional to rank_e^-s and rank a random permutation.
        rank = torch.randperm(E, generator=gen).to(torch.float64) + 1.0
        logp = (-cfg.zipf_s * torch.log(rank))
        logp = logp - torch.logsumexp(logp, 0)
        u = torch.rand((T, E), generator=gen, dtype=torch.float64).clamp_(1e-12, 1 - 1e-12)
        gumbel = -torch.log(-torch.log(u))
        return (logp[None, :] + gumbel).to(torch.float32)
    raise ValueError(cfg.logits)


def make_workload(cfg: LayerConfig, seed: int | None = None, weights: bool = True) -> Workload:
    """Draw one workload. ``weights=False`` skips the expert weights."""
    if seed is None:
        seed = CONFIG_SEEDS.get(cfg.key.split("-")[0], 1000)
    gen = torch.Generator().manual_seed(seed)
    dt = cfg.torch_dtype
    logits = [_logits(cfg, gen) for _ in range(cfg.layers)]
    X = _randn(gen, (cfg.T, cfg.H), cfg.x_std, dt)
    layers = []
    if weights:
        for _ in range(cfg.layers):
            Wg = torch.empty((cfg.E, cfg.F, cfg.H), dtype=dt)
            Wu = torch.empty((cfg.E, cfg.F, cfg.H), dtype=dt)
            Wd = torch.empty((cfg.E, cfg.H, cfg.F), dtype=dt)
            for e in range(cfg.E):
                Wg[e] = _randn(gen, (cfg.F, cfg.H), cfg.w_std, dt)
                Wu[e] = _randn(gen, (cfg.F, cfg.H), cfg.w_std, dt)
                Wd[e] = _randn(gen, (cfg.H, cfg.F), cfg.w_std, dt)
            Sg = Su = Sd = None
            if cfg.n_shared:
                Sg = _randn(gen, (cfg.n_shared, cfg.F_shared, cfg.H), cfg.w_std, dt)
                Su = _randn(gen, (cfg.n_shared, cfg.F_shared, cfg.H), cfg.w_std, dt)
                Sd = _randn(gen, (cfg.n_shared, cfg.H, cfg.F_shared), cfg.w_std, dt)
            layers.append(LayerWeights(Wg, Wu, Wd, Sg, Su, Sd))
    return Workload(cfg, logits, X, layers)


def random_permutation(E: int, seed: int) -> torch.Tensor:
    """A seeded storage order pi (int32)."""
    gen = torch.Generator().manual_seed(seed)
    return torch.randperm(E, generator=gen).to(torch.int32)


def sample_rows(T: int, n: int, seed: int = 7) -> torch.Tensor:
    """Seeded sorted sample of n distinct token rows (always includes the
    first and the last)."""
    n = min(n, T)
    gen = torch.Generator().manual_seed(seed)
    rows = torch.randperm(T, generator=gen)[:n]
    rows = torch.unique(torch.cat([rows, torch.tensor([0, T - 1])]))
    return rows.to(torch.int32)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def log2_ceil(x: int) -> int:
    return int(math.ceil(math.log2(max(1, x))))
