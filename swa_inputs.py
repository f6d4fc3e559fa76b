"""Seeded synthetic inputs for sliding-window attention, shared by the tests, the bench and smoke().

This module holds shapes and random-number draws only; it contains none of the attention
arithmetic. Both the fp64 oracle and the CUDA library take the tensors it returns.

Workload shapes follow the pages this library is built from:
  * Gemma 4 31B sliding-window layers: 32 query / 16 KV heads, window 1,024
    ("Off NVIDIA, you fix the platform yourself", section "What was broken?"; the lab record's
    numbers entry "Attention backward memory").  Head dim 128 is used here (the lab ran 256).
  * mlx-train-perf README, flash-attention section: batch 1, 32 query / 8 KV heads, 8,192 tokens,
    head_dim 128, full causal.
  * Longest training example: 30,553 tokens (the lab record's "load" field).
The pages' data (agent transcripts, trained weights) is not used: Gaussian bf16 tensors of the same
shapes stand in for the activations.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional

import torch

# Per-tensor seed offsets: every tensor of a case draws from its own generator.
_OFFSETS = {"q": 0, "k": 1, "v": 2, "do": 3}


@dataclasses.dataclass(frozen=True)
class Case:
    """One attention problem: [B, H, N, D] bf16 tensors, causal window W, softmax scale."""
    B: int
    Hq: int
    Hkv: int
    N: int
    D: int
    W: int
    do_std: float = 1.0
    seed: int = 0
    scale: Optional[float] = None

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def name(self) -> str:
        return f"B{self.B}_Hq{self.Hq}_Hkv{self.Hkv}_N{self.N}_D{self.D}_W{self.W}_s{self.seed}"


def _gaussian(shape, seed: int, std: float, device: str,
              dtype: torch.dtype = torch.bfloat16) -> torch.Tensor:
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def make_inputs(case: Case, device: str = "cpu", with_do: bool = True,
                dtype: torch.dtype = torch.bfloat16) -> Dict[str, torch.Tensor]:
    """Return {'q','k','v'[, 'do']} as contiguous tensors in [B, H, N, D] layout, bf16 unless
    `dtype` says otherwise (the same fp32 draws, rounded to fp16 or bf16, or kept as drawn for
    fp32).

    The same (case, device) always gives the same values.  CPU and CUDA generators give
    different streams, so the tests draw on the CPU and copy to the GPU when the oracle is
    compared against the device path.
    """
    base = case.seed * 16
    out = {
        "q": _gaussian((case.B, case.Hq, case.N, case.D), base + _OFFSETS["q"], 1.0, device, dtype),
        "k": _gaussian((case.B, case.Hkv, case.N, case.D), base + _OFFSETS["k"], 1.0, device, dtype),
        "v": _gaussian((case.B, case.Hkv, case.N, case.D), base + _OFFSETS["v"], 1.0, device, dtype),
    }
    if with_do:
        out["do"] = _gaussian((case.B, case.Hq, case.N, case.D), base + _OFFSETS["do"],
                              case.do_std, device, dtype)
    return out


# ---------------------------------------------------------------------------------------------
# Named workloads.
# ---------------------------------------------------------------------------------------------

def tiny_case() -> Case:
    """Tiny sliding-window check: one KV group of two query heads, 256 tokens, window 64."""
    return Case(B=1, Hq=2, Hkv=1, N=256, D=64, W=64)


def edge_cases() -> List[Case]:
    """Edge sweep: lengths that are not tile multiples, one-token windows, window == length."""
    cases = []
    for N in (1, 17, 128, 255, 512):
        for D in (64, 128):
            for W in (1, 7, 64, N):
                cases.append(Case(B=2, Hq=4, Hkv=2, N=N, D=D, W=W))
    # W == N duplicates W == 1 / 7 / 64 for short N; keep the list unique and ordered.
    seen, uniq = set(), []
    for c in cases:
        if c not in seen:
            seen.add(c)
            uniq.append(c)
    return uniq


def long_swa_case(N: int = 32768) -> Case:
    """Long-context sliding-window layer: 32 q / 16 kv heads, D 128, window 1,024, dO ~ N(0, 1e-2)."""
    return Case(B=1, Hq=32, Hkv=16, N=N, D=128, W=1024, do_std=1e-2)


def gqa_causal_case() -> Case:
    """Full-causal grouped-query layer: 32 q / 8 kv heads, 8,192 tokens, D 128, window = length."""
    return Case(B=1, Hq=32, Hkv=8, N=8192, D=128, W=8192)


MIXED_LAYERS = 12
MIXED_N = 30553


def mixed_layer_cases() -> List[Case]:
    """Mixed-layer step: 12 layers, five sliding (W=1,024) then one full-causal, repeated.

    Layer l is full-causal iff (l + 1) % 6 == 0, i.e. layers 5 and 11.  Each layer draws fresh
    inputs (seed = layer index + 1).
    """
    out = []
    for layer in range(MIXED_LAYERS):
        full = (layer + 1) % 6 == 0
        out.append(Case(B=1, Hq=32, Hkv=16, N=MIXED_N, D=128, W=MIXED_N if full else 1024, seed=layer + 1))
    return out

