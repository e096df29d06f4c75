"""Seeded synthetic inputs shaped like the pages' MoE workloads.

This module only draws random tensors; it holds none of the layer's
arithmetic (no gating, routing, expert or loss computation).  Both the
CUDA path (through the tests and ``bench.py``) and the fp64 oracle receive
the very same tensors from here, so a parity test compares the two
implementations on identical bits.

Shapes follow the 1 Billion Word layer of "Mixture of Experts: Outrageously
Large Neural Networks" (intuitivepapers.ai), section "How a mixture-of-experts
layer works": input/output size d = 512, hidden size h = 1024, k = 4 experts
per token, n from 32 to 4096 experts (section "What the paper measured").
The datasets themselves (1B Word, 100B Word, WMT'14) are not used; seeded
Gaussian tensors of the same shapes stand in for the layer's inputs:

* x ~ N(0, 1), rounded to bf16 for the bf16 workloads;
* W_g, W_noise, W_in ~ N(0, 1/d); W_out ~ N(0, 1/h) (variance 1/fan_in);
* eps ~ N(0, 1), one draw per (token, expert), supplied by the caller;
* the skewed 4096-expert workload adds a per-expert logit bias
  b_g[i] = ln p_{r(i)} with Zipf(s = 1.1) probabilities p_r over the ranks
  r = 1..n and r(i) a seeded permutation, so routing is heavy-tailed and
  some experts receive no token.

Random numbers come from torch's seeded generators: CPU draws for the small
cases, device draws for the multi-gigabyte expert weights of the large ones
(the oracle then receives a host copy of the same tensors).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch

__all__ = [
    "FlatShape",
    "HierShape",
    "WORKLOADS",
    "make_flat_inputs",
    "make_hier_inputs",
    "make_routing",
    "make_expert_rows",
]


@dataclasses.dataclass(frozen=True)
class FlatShape:
    """One flat MoE workload: T tokens, d model size, n experts, h hidden, k."""

    name: str
    T: int
    d: int
    n: int
    h: int
    k: int
    x_dtype: torch.dtype = torch.bfloat16
    expert_dtype: torch.dtype = torch.bfloat16
    zipf_bias: bool = False

    @property
    def R(self) -> int:
        return self.T * self.k


@dataclasses.dataclass(frozen=True)
class HierShape:
    """A two-level MoE: a groups of b experts, k1 groups then k2 experts each."""

    name: str
    T: int
    d: int
    a: int
    b: int
    h: int
    k1: int
    k2: int
    x_dtype: torch.dtype = torch.bfloat16
    expert_dtype: torch.dtype = torch.bfloat16


WORKLOADS = {
    # tiny, all fp32
    "tiny-fp32": FlatShape("tiny-fp32", 256, 64, 8, 128, 2, torch.float32, torch.float32),
    # 32 experts, the pages' LM layer shape
    "moe32": FlatShape("moe32", 16384, 512, 32, 1024, 4),
    # 256 experts, ~512 routed rows per expert
    "moe256": FlatShape("moe256", 32768, 512, 256, 1024, 4),
    # 4096 experts with Zipf-skewed routing (shrinking batch)
    "moe4096-zipf": FlatShape("moe4096-zipf", 65536, 512, 4096, 1024, 4, zipf_bias=True),
    # 128 groups x 128 experts, k = 2 x 2
    "hier128x128": HierShape("hier128x128", 65536, 512, 128, 128, 1024, 2, 2),
}


def _gen(device: str, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


_CHUNK = 1 << 28      # draw tensors above this many elements slab by slab


def _normal(shape, std: float, dtype: torch.dtype, device: str, g: torch.Generator) -> torch.Tensor:
    numel = math.prod(shape)
    if numel <= _CHUNK or dtype == torch.float32:
        t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        return t.to(dtype)
    # large low-precision tensors (the 16384-expert weights): fp32 draws one slab of
    # the leading dimension at a time, so no full-size fp32 copy is ever held
    out = torch.empty(shape, dtype=dtype, device=device)
    per = max(1, _CHUNK // (numel // shape[0]))
    for i in range(0, shape[0], per):
        j = min(shape[0], i + per)
        t = torch.randn((j - i,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        out[i:j] = t.to(dtype)
    return out


def zipf_logit_bias(n: int, s: float, seed: int) -> torch.Tensor:
    """ln of Zipf(s) probabilities over ranks 1..n, assigned to experts by a
    seeded permutation.  Returns a float32 tensor of n entries."""
    ranks = torch.arange(1, n + 1, dtype=torch.float64)
    w = ranks.pow(-s)
    p = w / w.sum()
    perm = torch.randperm(n, generator=_gen("cpu", seed ^ 0x5A17))
    bias = torch.empty(n, dtype=torch.float64)
    bias[perm] = p.log()
    return bias.to(torch.float32)


def make_flat_inputs(shape: FlatShape, seed: int = 0, device: str = "cpu",
                     zero_gate: bool = False, noise: bool = True) -> dict:
    """Draw every input of one flat MoE forward pass.

    Returns a dict with x[T,d], W_g[d,n], W_noise[d,n], eps[T,n] (fp32),
    b_g[n] or None, W_in[n,d,h], W_out[n,h,d], all contiguous on ``device``.
    ``zero_gate`` zero-initialises W_g and W_noise (the pages' start of
    training); ``noise=False`` passes eps = 0 (inference).
    """
    T, d, n, h = shape.T, shape.d, shape.n, shape.h
    g = _gen(device, seed)
    x = _normal((T, d), 1.0, shape.x_dtype, device, g)
    if zero_gate:
        W_g = torch.zeros((d, n), dtype=torch.float32, device=device)
        W_noise = torch.zeros((d, n), dtype=torch.float32, device=device)
    else:
        W_g = _normal((d, n), 1.0 / math.sqrt(d), torch.float32, device, g)
        W_noise = _normal((d, n), 1.0 / math.sqrt(d), torch.float32, device, g)
    eps = _normal((T, n), 1.0, torch.float32, device, g)
    if not noise:
        eps.zero_()
    W_in = _normal((n, d, h), 1.0 / math.sqrt(d), shape.expert_dtype, device, g)
    W_out = _normal((n, h, d), 1.0 / math.sqrt(h), shape.expert_dtype, device, g)
    b_g: Optional[torch.Tensor] = None
    if shape.zipf_bias:
        b_g = zipf_logit_bias(n, 1.1, seed).to(device)
    return dict(x=x, W_g=W_g, W_noise=W_noise, eps=eps, b_g=b_g, W_in=W_in, W_out=W_out)


def make_hier_inputs(shape: HierShape, seed: int = 0, device: str = "cpu") -> dict:
    """Draw every input of one hierarchical MoE forward pass.

    x[T,d]; primary W_g1, W_noise1 [d,a]; secondary W_g2, W_noise2 [a,d,b];
    eps1[T,a]; eps2[T,k1,b] (one draw per chosen group slot);
    W_in[a*b,d,h], W_out[a*b,h,d].
    """
    T, d, a, b, h = shape.T, shape.d, shape.a, shape.b, shape.h
    g = _gen(device, seed)
    x = _normal((T, d), 1.0, shape.x_dtype, device, g)
    W_g1 = _normal((d, a), 1.0 / math.sqrt(d), torch.float32, device, g)
    W_noise1 = _normal((d, a), 1.0 / math.sqrt(d), torch.float32, device, g)
    W_g2 = _normal((a, d, b), 1.0 / math.sqrt(d), torch.float32, device, g)
    W_noise2 = _normal((a, d, b), 1.0 / math.sqrt(d), torch.float32, device, g)
    eps1 = _normal((T, a), 1.0, torch.float32, device, g)
    eps2 = _normal((T, shape.k1, b), 1.0, torch.float32, device, g)
    W_in = _normal((a * b, d, h), 1.0 / math.sqrt(d), shape.expert_dtype, device, g)
    W_out = _normal((a * b, h, d), 1.0 / math.sqrt(h), shape.expert_dtype, device, g)
    return dict(x=x, W_g1=W_g1, W_noise1=W_noise1, W_g2=W_g2, W_noise2=W_noise2,
                eps1=eps1, eps2=eps2, W_in=W_in, W_out=W_out)


def make_expert_rows(R: int, n: int, d: int, dtype: torch.dtype, seed: int = 0,
                     empty_experts: int = 0, skew: float = 0.0) -> tuple:
    """Draw expert-grouped rows for testing the expert FFN in isolation.

    Returns x_rows [R,d] ~ N(0,1) in ``dtype`` and offsets [n+1] int32 whose
    per-expert counts are a multinomial draw of R rows over the experts
    (weights rank**-skew, the last ``empty_experts`` experts get none).
    """
    g = _gen("cpu", seed)
    live = n - empty_experts
    w = torch.arange(1, live + 1, dtype=torch.float64).pow(-skew)
    w = w[torch.randperm(live, generator=g)]
    counts = torch.zeros(n, dtype=torch.int64)
    if R > 0:
        draws = torch.multinomial(w, R, replacement=True, generator=g)
        counts[:live] = torch.bincount(draws, minlength=live)
    offsets = torch.zeros(n + 1, dtype=torch.int32)
    offsets[1:] = torch.cumsum(counts, 0).to(torch.int32)
    x_rows = torch.randn((R, d), generator=g, dtype=torch.float32).to(dtype)
    return x_rows, offsets


def make_routing(T: int, n: int, k: int, seed: int = 0, skew: float = 0.0,
                 empty_experts: int = 0) -> tuple:
    """Draw a routing table for testing dispatch/combine in isolation.

    idx[T,k] int32 holds k distinct experts per token (a random draw without
    replacement, weighted by rank**-skew); the last ``empty_experts`` experts
    are never drawn.  gates[T,k] fp32 are positive and sum to 1 per row
    (normalised uniform draws, not a gate computation).
    """
    g = _gen("cpu", seed)
    live = n - empty_experts
    if k > live:
        raise ValueError("k exceeds the number of experts that may be drawn")
    w = torch.arange(1, live + 1, dtype=torch.float64).pow(-skew)
    w = w[torch.randperm(live, generator=g)]
    # draw with replacement, then redraw the rows that hold a repeated expert
    idx = torch.multinomial(w, T * k, replacement=True, generator=g).view(T, k)
    while k > 1:
        s, _ = idx.sort(dim=1)
        dup = (s[:, 1:] == s[:, :-1]).any(dim=1).nonzero().flatten()
        if dup.numel() == 0:
            break
        idx[dup] = torch.multinomial(w, dup.numel() * k, replacement=True, generator=g).view(-1, k)
    idx = idx.to(torch.int32)
    u = torch.rand((T, k), generator=g, dtype=torch.float64) + 0.05
    gates = (u / u.sum(dim=1, keepdim=True)).to(torch.float32)
    return idx.contiguous(), gates.contiguous()
