"""Seeded synthetic inputs for the MoE-layer forward.

This module holds no arithmetic of the method: it only draws random tensors
with the shapes and distributions of the workloads the MoE pages discuss
(the coarse-grained Mixtral shape and the fine-grained DeepSeek-V3 / 7B shapes
in the granularity table of "SonicMoE: 加速 MoE 模型的 IO 与 Tile 感知优化",
section "MoE 的两个核心趋势").  Both the CUDA path and the fp64 oracle are fed
from here, and from nowhere else.

Layouts (all row-major, contiguous):
  x    [T, d]    bf16   token activations
  Wr   [d, E]    fp32   router weight
  bias [E]       fp32   per-expert router logit bias, or None
  W1   [E, d, n] bf16   gated (silu) branch of the SwiGLU up-projection
  W3   [E, d, n] bf16   linear branch of the SwiGLU up-projection
  W2   [E, n, d] bf16   down-projection
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import torch


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    d: int
    n: int
    E: int
    k: int
    # std of x; the weight stds are 1/sqrt(fan_in) unless overridden below
    x_std: float = 1.0
    wr_std: float | None = None          # default 1/sqrt(d)
    w13_std: float | None = None         # default 1/sqrt(d)
    w2_std: float | None = None          # default 1/sqrt(n)
    bias: str | None = None              # None | "normal" | "zipf"
    bias_scale: float = 0.0              # std of the normal bias / Zipf exponent
    tile: int = 128                      # token-rounding tile
    description: str = ""

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T)

    @property
    def assignments(self) -> int:
        return self.T * self.k

    def active_flops(self) -> float:
        """Useful expert FLOPs: 2*T*k*(2*d*n) up + 2*T*k*n*d down."""
        return 6.0 * self.T * self.k * self.d * self.n

    def router_flops(self) -> float:
        return 2.0 * self.T * self.d * self.E


CONFIGS: dict[str, MoEConfig] = {
    "tiny": MoEConfig("tiny", T=256, d=128, n=64, E=8, k=2,
                      description="tiny MoE layer T=256 d=128 n=64 E=8 k=2"),
    "mixtral": MoEConfig("mixtral", T=8192, d=4096, n=14336, E=8, k=2,
                         bias="normal", bias_scale=0.1,
                         description="coarse-grained Mixtral-style layer T=8192 d=4096 n=14336 E=8 k=2, "
                                     "router bias ~N(0, 0.1^2)"),
    "dsv3": MoEConfig("dsv3", T=16384, d=7168, n=2048, E=256, k=8,
                      description="fine-grained DeepSeek-V3-style layer T=16384 d=7168 n=2048 E=256 k=8"),
    "b7": MoEConfig("b7", T=32768, d=1536, n=256, E=128, k=8,
                    description="fine-grained 7B-class layer T=32768 d=1536 n=256 E=128 k=8"),
    "skew": MoEConfig("skew", T=32768, d=4096, n=1024, E=128, k=8,
                      bias="zipf", bias_scale=1.1, tile=128,
                      description="skewed-load layer T=32768 d=4096 n=1024 E=128 k=8, "
                                  "Zipf(1.1) per-expert router bias"),
}


def get_config(name: str) -> MoEConfig:
    if name not in CONFIGS:
        raise KeyError(f"unknown config {name!r}; known: {sorted(CONFIGS)}")
    return CONFIGS[name]


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def make_inputs(cfg: MoEConfig, device="cpu", seed: int = 0, weights: bool = True) -> dict:
    """Draw x, Wr, bias and (optionally) W1, W3, W2 for `cfg` on `device`.

    The draw order is fixed (x, Wr, bias, W1, W3, W2), so a seed names one
    input set per device.  Weights are drawn one expert at a time to bound
    the fp32 temporaries at full size.
    """
    dev = torch.device(device)
    g = _gen(dev, seed)
    T, d, n, E = cfg.T, cfg.d, cfg.n, cfg.E
    x = (torch.randn(T, d, generator=g, device=dev) * cfg.x_std).to(torch.bfloat16)
    wr_std = cfg.wr_std if cfg.wr_std is not None else 1.0 / math.sqrt(d)
    Wr = torch.randn(d, E, generator=g, device=dev) * wr_std
    bias = None
    if cfg.bias == "normal":
        bias = torch.randn(E, generator=g, device=dev) * cfg.bias_scale
    elif cfg.bias == "zipf":
        # expert popularity proportional to rank^-s, ranks a seeded permutation
        # of 1..E: the logit bias is -s*ln(rank)
        rank = torch.randperm(E, generator=g, device=dev).to(torch.float32) + 1.0
        bias = -cfg.bias_scale * torch.log(rank)
    out = {"x": x, "Wr": Wr.contiguous(), "bias": bias}
    if weights:
        w13_std = cfg.w13_std if cfg.w13_std is not None else 1.0 / math.sqrt(d)
        w2_std = cfg.w2_std if cfg.w2_std is not None else 1.0 / math.sqrt(n)
        W1 = torch.empty(E, d, n, dtype=torch.bfloat16, device=dev)
        W3 = torch.empty(E, d, n, dtype=torch.bfloat16, device=dev)
        W2 = torch.empty(E, n, d, dtype=torch.bfloat16, device=dev)
        for e in range(E):
            W1[e] = (torch.randn(d, n, generator=g, device=dev) * w13_std).to(torch.bfloat16)
        for e in range(E):
            W3[e] = (torch.randn(d, n, generator=g, device=dev) * w13_std).to(torch.bfloat16)
        for e in range(E):
            W2[e] = (torch.randn(n, d, generator=g, device=dev) * w2_std).to(torch.bfloat16)
        out.update(W1=W1, W3=W3, W2=W2)
    return out


def make_replica_inputs(cfg: MoEConfig, rank: int, device="cpu") -> dict:
    """Inputs of one data-parallel replica: every rank holds the same layer
    (x, Wr, bias and weights drawn with seed 0, as make_inputs) and rank r > 0
    replaces x with its own tokens, drawn from the same distribution with
    seed 1_000_003 * r."""
    out = make_inputs(cfg, device=device, seed=0)
    if rank > 0:
        g = _gen(torch.device(device), 1_000_003 * rank)
        out["x"] = (torch.randn(cfg.T, cfg.d, generator=g, device=device) * cfg.x_std).to(torch.bfloat16)
    return out


def make_logits(T: int, E: int, device="cpu", seed: int = 0, ties: bool = True) -> torch.Tensor:
    """fp32 router logits [T, E].  With `ties`, values sit on a coarse grid
    (multiples of 1/4, including both signed zeros) so equal logits are common."""
    g = _gen(torch.device(device), seed)
    L = torch.randn(T, E, generator=g, device=device)
    if ties:
        L = torch.round(L * 4.0) / 4.0
        # sprinkle negative zeros next to positive ones
        neg = torch.rand(T, E, generator=g, device=device) < 0.5
        L = torch.where((L == 0) & neg, torch.full_like(L, -0.0), L)
    return L.contiguous()


def make_topk_idx(T: int, E: int, k: int, device="cpu", seed: int = 0, skew: float = 0.0) -> torch.Tensor:
    """int32 [T, k] expert ids, distinct within a row.  `skew` > 0 draws
    experts with Zipf-like popularity so some experts get far more rows."""
    g = _gen(torch.device(device), seed)
    if skew > 0:
        w = (torch.arange(1, E + 1, dtype=torch.float64, device=device) ** (-skew)).float()
        w = w.expand(T, E)
        idx = torch.multinomial(w, k, replacement=False, generator=g)
    else:
        idx = torch.rand(T, E, generator=g, device=device).argsort(dim=1)[:, :k]
    return idx.to(torch.int32).contiguous()


def make_gate_weights(T: int, k: int, device="cpu", seed: int = 0) -> torch.Tensor:
    """fp32 [T, k] positive weights (any values; the permutation only moves them)."""
    g = _gen(torch.device(device), seed)
    return torch.rand(T, k, generator=g, device=device).contiguous()
