"""Seeded synthetic inputs for the block-FP8 MoE layer.

This module is shared by the tests, the benchmark and the oracle's callers.  It
holds no arithmetic of the method (no quantisation, routing or GEMM): it only
draws random tensors with the shapes and value distributions of the
workloads, from torch's seeded generators.

Workloads (model-shaped MoE layers, all with 128x128 block-FP8 weights and
1x128 dynamic activation groups):

  tiny        T=16    H=256  I=256   E=4   k=2  softmax + renormalize
  mixtral     T=512   H=4096 I=14336 E=8   k=2  softmax + renormalize
  dsv3        T=4096  H=7168 I=2048  E=256 k=8  sigmoid + bias N(0,0.01), n_group=8,
                                                 topk_group=4, renormalize, scaling 2.5
  dsv3_decode T in {1,8,32,64,128}, otherwise dsv3
  qwen3_skew  T=16384 H=2048 I=768   E=128 k=8  softmax + renormalize, logits
                                                 N(0,1) - 1.2*ln(e+1) (Zipf s=1.2)

Hidden states are bf16 N(0,1), router logits fp32 N(0,1), expert weights bf16
N(0,0.02) (quantised to e4m3 blocks by the caller: each side of a parity test
quantises its own copy).  Seeds: 1000 + workload number, with a fixed offset
per tensor so that each tensor can be regenerated alone.
"""
from __future__ import annotations

import dataclasses
import math

import torch

SOFTMAX, SIGMOID = 0, 1


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    number: int
    T: int
    H: int
    I: int
    E: int
    topk: int
    scoring: int = SOFTMAX
    renormalize: bool = True
    n_group: int = 1
    topk_group: int = 1
    routed_scaling: float = 1.0
    bias_std: float = 0.0
    zipf_s: float = 0.0

    @property
    def seed(self) -> int:
        return 1000 + self.number

    @property
    def P(self) -> int:
        return self.T * self.topk

    def with_tokens(self, T: int) -> "Workload":
        return dataclasses.replace(self, T=T)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def flops(self) -> int:
        """Dense work of the two grouped GEMMs: 2*P*H*(2I) + 2*P*I*H."""
        return 6 * self.P * self.H * self.I

    def describe(self) -> dict:
        d = dataclasses.asdict(self)
        d["scoring"] = "sigmoid" if self.scoring == SIGMOID else "softmax"
        return d


WORKLOADS = {
    "tiny": Workload("tiny", 1, T=16, H=256, I=256, E=4, topk=2),
    "mixtral": Workload("mixtral", 2, T=512, H=4096, I=14336, E=8, topk=2),
    "dsv3": Workload("dsv3", 3, T=4096, H=7168, I=2048, E=256, topk=8, scoring=SIGMOID,
                     n_group=8, topk_group=4, routed_scaling=2.5, bias_std=0.01),
    "dsv3_decode": Workload("dsv3_decode", 4, T=128, H=7168, I=2048, E=256, topk=8, scoring=SIGMOID,
                            n_group=8, topk_group=4, routed_scaling=2.5, bias_std=0.01),
    "qwen3_skew": Workload("qwen3_skew", 5, T=16384, H=2048, I=768, E=128, topk=8, zipf_s=1.2),
}
DECODE_TOKENS = (1, 8, 32, 64, 128)

# tensor ids: part of the seed so that each tensor regenerates independently
_HIDDEN, _LOGITS, _BIAS, _W13, _W2 = 1, 2, 3, 4, 5


def _gen(seed: int, tensor: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + tensor * 7919)
    return g


def hidden(wl: Workload, device="cpu") -> torch.Tensor:
    """bf16 [T, H] ~ N(0, 1)."""
    g = _gen(wl.seed, _HIDDEN, device)
    return torch.randn(wl.T, wl.H, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def router_logits(wl: Workload, device="cpu") -> torch.Tensor:
    """fp32 [T, E] ~ N(0, 1), plus -s*ln(e+1) per expert for a Zipf(s) popularity."""
    g = _gen(wl.seed, _LOGITS, device)
    x = torch.randn(wl.T, wl.E, generator=g, device=device, dtype=torch.float32)
    if wl.zipf_s:
        offs = torch.tensor([-wl.zipf_s * math.log(e + 1.0) for e in range(wl.E)], dtype=torch.float32)
        x = x + offs.to(device)
    return x


def expert_bias(wl: Workload, device="cpu") -> torch.Tensor | None:
    """fp32 [E] ~ N(0, bias_std), or None when the workload has no selection bias."""
    if not wl.bias_std:
        return None
    g = _gen(wl.seed, _BIAS, device)
    return torch.randn(wl.E, generator=g, device=device, dtype=torch.float32) * wl.bias_std


def _expert_stack(wl: Workload, tensor: int, N: int, K: int, device, experts=None) -> torch.Tensor:
    """bf16 [len(experts), N, K] ~ N(0, 0.02); expert e is drawn from its own stream so that any
    subset regenerates identically on the same device type."""
    experts = range(wl.E) if experts is None else list(experts)
    out = torch.empty(len(experts), N, K, dtype=torch.bfloat16, device=device)
    for i, e in enumerate(experts):
        g = _gen(wl.seed, tensor * 100_003 + e, device)
        out[i] = (torch.randn(N, K, generator=g, device=device, dtype=torch.float32) * 0.02).to(torch.bfloat16)
    return out


def w13_bf16(wl: Workload, device="cpu", experts=None) -> torch.Tensor:
    """bf16 [E, 2I, H]: rows [0, I) gate projection, rows [I, 2I) up projection."""
    return _expert_stack(wl, _W13, 2 * wl.I, wl.H, device, experts)


def w2_bf16(wl: Workload, device="cpu", experts=None) -> torch.Tensor:
    """bf16 [E, H, I]: down projection."""
    return _expert_stack(wl, _W2, wl.H, wl.I, device, experts)


def bf16_bits(t: torch.Tensor):
    """numpy uint16 view of a bf16 tensor's bits (copied to the host)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view("uint16")
