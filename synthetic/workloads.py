"""Seeded synthetic inputs for the routed-MoE forward with per-token NVFP4.

Shapes and value distributions follow the workloads the pages describe (a
decode batch, a speculative-decode batch with skewed routing, a prefill chunk
at the worst-case buffer size, and a per-token-scale stress case with an
in-place weight reload).  There is no dataset or checkpoint behind any of
them: every tensor is drawn from ``torch.Generator`` streams on the CPU, one
stream per tensor so that changing the token count never changes the weights.

Everything returned is a CPU tensor in the dtype the library consumes:
bf16 activations and weights, and an fp32 per-expert router bias.
"""

from __future__ import annotations

import dataclasses
from typing import Optional, Tuple

import torch

# One generator stream per tensor kind.
_TAG_X, _TAG_GATE, _TAG_W13, _TAG_W2, _TAG_BIAS, _TAG_ROWS = 1, 2, 3, 4, 5, 6
_TAG_SW13, _TAG_SW2 = 7, 8


def _gen(seed: int, tag: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) * 1_000_003 + tag)
    return g


@dataclasses.dataclass(frozen=True)
class MoEShape:
    """Sizes of one MoE layer and of one forward through it.

    T tokens, H hidden size, E experts, K experts per token (top-k),
    I expert intermediate size (w13 is [E, 2I, H], w2 is [E, H, I]).
    """

    name: str
    T: int
    H: int
    E: int
    K: int
    I: int
    max_num_tokens: int
    deterministic: bool = False
    zipf_bias: bool = False
    x_kind: str = "normal"          # "normal" or "stress"
    token_sweep: Tuple[int, ...] = ()
    refresh_seed: Optional[int] = None
    graph: bool = False

    @property
    def rows(self) -> int:
        """Expanded rows R = T*K of one forward."""
        return self.T * self.K


CONFIGS = {
    # Tiny layer: small enough for the oracle's pure-Python checks.
    "c0_tiny": MoEShape("c0_tiny", T=16, H=256, E=8, K=2, I=128, max_num_tokens=16),
    # Decode-shaped batch: ~4 rows per expert, weight streaming dominates.
    "c1_decode": MoEShape("c1_decode", T=64, H=2048, E=128, K=8, I=768,
                          max_num_tokens=64, graph=True),
    # Speculative decode: 64 sequences x 4 draft tokens, Zipf-skewed routing,
    # deterministic (fixed-order) finalize.
    "c2_specdecode": MoEShape("c2_specdecode", T=256, H=2048, E=128, K=8, I=768,
                              max_num_tokens=256, deterministic=True, zipf_bias=True),
    # Prefill chunk on an instance sized for the worst case of 4096 tokens.
    "c3_prefill": MoEShape("c3_prefill", T=4096, H=2048, E=128, K=8, I=768,
                           max_num_tokens=4096, token_sweep=(1, 17, 2048, 4073, 4096)),
    # Per-token-scale stress: row norms over six decades, zero rows, outlier
    # channels; weights redrawn from a second seed for the in-place reload.
    "c4_stress": MoEShape("c4_stress", T=2048, H=4096, E=64, K=6, I=1536,
                          max_num_tokens=2048, deterministic=True, x_kind="stress",
                          refresh_seed=1, graph=True),
}


def make_activations(shape: MoEShape, T: Optional[int] = None, seed: int = 0) -> torch.Tensor:
    """Token activations x, bf16 [T, H].

    "normal": i.i.d. N(0, 1).
    "stress": each row is a N(0,1) vector rescaled to an L2 norm of 10**u with
    u ~ U[-3, 3]; 8 seeded channels are multiplied by 100 in every row; 1% of
    the rows (seeded) are all zero.
    """
    T = shape.T if T is None else int(T)
    g = _gen(seed, _TAG_X)
    z = torch.randn(T, shape.H, generator=g, dtype=torch.float32)
    if shape.x_kind == "stress" and T > 0:
        u = torch.rand(T, generator=g, dtype=torch.float64) * 6.0 - 3.0
        norms = z.double().norm(dim=1).clamp_min(1e-30)
        z = (z.double() * (torch.pow(10.0, u) / norms)[:, None])
        channels = torch.randperm(shape.H, generator=g)[:8]
        z[:, channels] *= 100.0
        n_zero = int(round(0.01 * T))
        zero_rows = torch.randperm(T, generator=g)[:n_zero]
        z[zero_rows] = 0.0
        z = z.float()
    elif shape.x_kind != "normal":
        raise ValueError(f"unknown activation kind {shape.x_kind!r}")
    return z.to(torch.bfloat16)


def make_router(shape: MoEShape, seed: int = 0) -> torch.Tensor:
    """Router (gate) weight Wg, bf16 [H, E], N(0, 0.02)."""
    g = _gen(seed, _TAG_GATE)
    return (torch.randn(shape.H, shape.E, generator=g, dtype=torch.float32) * 0.02).to(torch.bfloat16)


def zipf_router_bias(shape: MoEShape, seed: int = 0, s: float = 1.2) -> torch.Tensor:
    """Per-expert router-logit bias b_e = -s * ln(rank_e), fp32 [E].

    rank is a seeded permutation of 1..E, so a Zipf(s) prior lands on random
    experts: a few experts draw most rows and several draw none.
    """
    g = _gen(seed, _TAG_BIAS)
    rank = (torch.randperm(shape.E, generator=g) + 1).double()
    return (-s * torch.log(rank)).float()


def make_weights(shape: MoEShape, seed: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Expert weights w13 bf16 [E, 2I, H] and w2 bf16 [E, H, I], N(0, 0.02).

    Rows [0, I) of w13[e] are the gate projection (w1), rows [I, 2I) the up
    projection (w3).  Drawn one expert at a time to bound peak host memory.
    """
    E, H, I = shape.E, shape.H, shape.I
    w13 = torch.empty(E, 2 * I, H, dtype=torch.bfloat16)
    w2 = torch.empty(E, H, I, dtype=torch.bfloat16)
    g13 = _gen(seed, _TAG_W13)
    g2 = _gen(seed, _TAG_W2)
    for e in range(E):
        w13[e] = (torch.randn(2 * I, H, generator=g13, dtype=torch.float32) * 0.02).to(torch.bfloat16)
        w2[e] = (torch.randn(H, I, generator=g2, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return w13, w2


def make_shared_weights(shape: MoEShape, shared_inter: int, seed: int = 0) -> Tuple[torch.Tensor, torch.Tensor]:
    """Shared-expert weights w13s bf16 [2*Is, H] (gate rows, then up rows) and
    w2s bf16 [H, Is], N(0, 0.02), from streams of their own."""
    H, Is = shape.H, shared_inter
    w13s = (torch.randn(2 * Is, H, generator=_gen(seed, _TAG_SW13), dtype=torch.float32) * 0.02).to(torch.bfloat16)
    w2s = (torch.randn(H, Is, generator=_gen(seed, _TAG_SW2), dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return w13s, w2s


@dataclasses.dataclass
class Workload:
    shape: MoEShape
    x: torch.Tensor                 # bf16 [T, H]
    gate_w: torch.Tensor            # bf16 [H, E]
    w13: torch.Tensor               # bf16 [E, 2I, H]
    w2: torch.Tensor                # bf16 [E, H, I]
    bias: Optional[torch.Tensor]    # fp32 [E] or None

    @property
    def T(self) -> int:
        return int(self.x.shape[0])


def make_workload(name_or_shape, T: Optional[int] = None, seed: int = 0,
                  weight_seed: Optional[int] = None) -> Workload:
    """Build the full input set of one configuration.

    ``T`` overrides the token count (the prefill sweep); ``weight_seed``
    redraws only the expert weights (the in-place reload case).
    """
    shape = CONFIGS[name_or_shape] if isinstance(name_or_shape, str) else name_or_shape
    if T is not None and T > shape.max_num_tokens:
        raise ValueError(f"T={T} exceeds the configuration's max_num_tokens={shape.max_num_tokens}")
    x = make_activations(shape, T=T, seed=seed)
    gate_w = make_router(shape, seed=seed)
    w13, w2 = make_weights(shape, seed=seed if weight_seed is None else weight_seed)
    bias = zipf_router_bias(shape, seed=seed) if shape.zipf_bias else None
    return Workload(shape=shape, x=x, gate_w=gate_w, w13=w13, w2=w2, bias=bias)


def expected_zero_rows(shape: MoEShape, T: int) -> int:
    """How many all-zero rows the stress activations contain (for tests)."""
    return int(round(0.01 * T)) if shape.x_kind == "stress" else 0


__all__ = ["CONFIGS", "MoEShape", "Workload", "make_activations", "make_router",
           "make_weights", "make_workload", "zipf_router_bias", "expected_zero_rows"]
