"""Seeded synthetic inputs for the FP4 quantized linear layer.

This module only draws random numbers and converts them to BF16 bit patterns.
It holds none of the method's arithmetic (no scales, no rounding to E2M1, no
quantile, no GEMM), so that the CPU oracle and the CUDA library can both be fed
the same bytes without sharing any code.

Shapes follow the LLaMA model sizes named on the pages (1.3B / 7B / 13B, see
"Optimizing Large Language Model Training Using FP4 Quantization", abstract);
the pages train on a dataset they do not name, which is not available here, so
these draws stand in for activations, weights and output gradients:

* activations ~ N(0, 1) with a seeded 0.5 % of channels made into outliers
  (x20 for the 7B/13B decoder layers, redrawn ~N(0, 15^2) for the 1.3B MLP),
* weights ~ N(0, 0.02), output gradients ~ N(0, 1e-3) (std, not variance),
* the outlier-stress case draws Student-t with 3 degrees of freedom.

Every tensor gets its own independent PCG64 stream derived from the config
seed, so a tensor can be regenerated without drawing the others.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, List, Tuple

import numpy as np
import torch

__all__ = [
    "LinearCase", "Workload", "WORKLOADS", "f32_to_bf16_bits", "bf16_bits_to_f32_view",
    "draw_activation", "draw_weight", "draw_grad", "outlier_channels", "fuse_shared_inputs", "FusedWorkload",
]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round an fp32 array to BF16 (torch's round-to-nearest-even) and return the uint16 bits."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32_view(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to fp32 values (exact: BF16 is the top half of fp32)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def _rng(seed: int, stream: str) -> np.random.Generator:
    # One independent stream per (seed, tensor name): stable across calls.
    key = [seed] + [ord(c) for c in stream]
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(key)))


def outlier_channels(seed: int, name: str, K: int, frac: float = 0.005) -> np.ndarray:
    """Seeded choice of max(1, round(frac*K)) channel indices (sorted)."""
    n_out = max(1, int(round(frac * K)))
    perm = _rng(seed, name + "/outlier_channels").permutation(K)
    return np.sort(perm[:n_out])


def draw_activation(seed: int, name: str, M: int, K: int, kind: str, rows: int | None = None) -> np.ndarray:
    """Activation A (M x K) as BF16 bits, or only its first `rows` rows.

    kind = "normal_x20"       N(0,1), 0.5 % of channels multiplied by 20
           "normal_redraw15"  N(0,1), 0.5 % of channels redrawn ~N(0, 15^2)
           "normal_4x20"      N(0,1), 4 channels multiplied by 20
           "student_t3"       Student-t, 3 degrees of freedom, per element

    Every stream is consumed in row-major order, so the first `rows` rows are
    the same values as the first rows of the whole draw.
    """
    M = M if rows is None else min(M, rows)
    rng = _rng(seed, name)
    if kind == "student_t3":
        x = rng.standard_t(3, size=(M, K)).astype(np.float32)
        return f32_to_bf16_bits(x)
    x = rng.standard_normal(size=(M, K), dtype=np.float32)
    if kind == "normal_x20":
        ch = outlier_channels(seed, name, K)
        x[:, ch] *= np.float32(20.0)
    elif kind == "normal_redraw15":
        ch = outlier_channels(seed, name, K)
        x[:, ch] = _rng(seed, name + "/redraw").standard_normal(size=(M, ch.size), dtype=np.float32) * np.float32(15.0)
    elif kind == "normal_4x20":
        ch = np.sort(_rng(seed, name + "/outlier_channels").permutation(K)[:4])
        x[:, ch] *= np.float32(20.0)
    elif kind != "normal":
        raise ValueError(f"unknown activation kind {kind!r}")
    return f32_to_bf16_bits(x)


def draw_weight(seed: int, name: str, K: int, N: int, std: float = 0.02) -> np.ndarray:
    """Weight W (K x N, in-features x out-features, row-major) as BF16 bits."""
    x = _rng(seed, name).standard_normal(size=(K, N), dtype=np.float32) * np.float32(std)
    return f32_to_bf16_bits(x)


def draw_grad(seed: int, name: str, M: int, N: int, std: float = 1e-3, rows: int | None = None) -> np.ndarray:
    """Output gradient dY (M x N) as BF16 bits, or only its first `rows` rows."""
    M = M if rows is None else min(M, rows)
    x = _rng(seed, name).standard_normal(size=(M, N), dtype=np.float32) * np.float32(std)
    return f32_to_bf16_bits(x)


@dataclasses.dataclass(frozen=True)
class LinearCase:
    """One linear layer Y = A W with A: M x K (tokens x in), W: K x N (in x out)."""
    name: str
    M: int
    K: int
    N: int
    act: str        # name of the activation tensor (linears sharing it share A)
    act_kind: str   # distribution, see draw_activation
    q: float        # clamp quantile of |A|
    weight_name: str = ""  # linears with the same weight_name share W (default: own name)

    @property
    def flops_fwd(self) -> int:
        return 2 * self.M * self.K * self.N


@dataclasses.dataclass(frozen=True)
class Workload:
    key: str
    seed: int
    description: str
    linears: Tuple[LinearCase, ...]

    def activation(self, lin: LinearCase, rows: int | None = None) -> np.ndarray:
        return draw_activation(self.seed, lin.act, lin.M, lin.K, lin.act_kind, rows=rows)

    def weight(self, lin: LinearCase) -> np.ndarray:
        return draw_weight(self.seed, "W/" + (lin.weight_name or lin.name), lin.K, lin.N)

    def grad(self, lin: LinearCase, rows: int | None = None) -> np.ndarray:
        return draw_grad(self.seed, "dY/" + lin.name, lin.M, lin.N, rows=rows)


def _decoder(key: str, seed: int, desc: str, M: int, H: int, F: int) -> Workload:
    kind = "normal_x20"
    lins = (
        LinearCase("q_proj", M, H, H, "x_attn", kind, 0.999),
        LinearCase("k_proj", M, H, H, "x_attn", kind, 0.999),
        LinearCase("v_proj", M, H, H, "x_attn", kind, 0.999),
        LinearCase("o_proj", M, H, H, "attn_out", kind, 0.999),
        LinearCase("gate_proj", M, H, F, "x_mlp", kind, 0.999),
        LinearCase("up_proj", M, H, F, "x_mlp", kind, 0.999),
        LinearCase("down_proj", M, F, H, "h_mlp", kind, 0.999),
    )
    return Workload(key, seed, desc, lins)


WORKLOADS: Dict[str, Workload] = {
    "c1_single_linear_256x512x512": Workload(
        "c1_single_linear_256x512x512", 0,
        "single FP4 linear, A 256x512 N(0,1) with 4 outlier columns x20, W 512x512 N(0,0.02), q=0.99",
        (LinearCase("linear", 256, 512, 512, "x", "normal_4x20", 0.99),)),
    "c2_llama1.3b_mlp_up_8192x2048x5504": Workload(
        "c2_llama1.3b_mlp_up_8192x2048x5504", 1,
        "LLaMA-1.3B MLP up-projection, A 8192x2048 with 0.5% channels ~N(0,15^2), W 2048x5504, q=0.999",
        (LinearCase("up_proj", 8192, 2048, 5504, "x_mlp", "normal_redraw15", 0.999),)),
    "c3_llama7b_layer_8192tok": _decoder(
        "c3_llama7b_layer_8192tok", 2, "LLaMA-7B decoder-layer linears, 8192 tokens, hidden 4096, FFN 11008",
        8192, 4096, 11008),
    "c4_llama13b_layer_16384tok": _decoder(
        "c4_llama13b_layer_16384tok", 3, "LLaMA-13B decoder-layer linears, 16384 tokens, hidden 5120, FFN 13824",
        16384, 5120, 13824),
    "c5_outlier_stress_16384x5120x5120": Workload(
        "c5_outlier_stress_16384x5120x5120", 4,
        "Student-t(3) activations 16384x5120, W 5120x5120, q in {0.97, 0.99, 0.999}",
        tuple(LinearCase(f"stress_q{q}", 16384, 5120, 5120, "x_t3", "student_t3", q, "stress")
              for q in (0.97, 0.99, 0.999))),
}

WORKLOAD_ORDER: List[str] = list(WORKLOADS)


class FusedWorkload:
    """A workload whose linears that read the same activation (and clamp
    quantile) are one linear over their weights placed side by side: W_cat =
    [W_1 | W_2 | ...] (K x sum N), dY_cat = [dY_1 | dY_2 | ...].  Only the layout
    of the inputs changes: Y_cat = A W_cat holds each member's Y as a column
    block, dW_cat each member's dW, and dY_cat W_cat^T = sum_i dY_i W_i^T is
    the summed input gradient of the shared activation."""

    def __init__(self, work: Workload):
        self.base = work
        self.key = work.key
        self.seed = work.seed
        groups: Dict[Tuple[str, float], List[LinearCase]] = {}
        for lin in work.linears:
            groups.setdefault((lin.act, lin.q), []).append(lin)
        self.members: Dict[str, Tuple[LinearCase, ...]] = {}
        fused = []
        for lins in groups.values():
            if len(lins) == 1:
                f = lins[0]
            else:
                name = "+".join(l.name for l in lins)
                f = dataclasses.replace(lins[0], name=name, N=sum(l.N for l in lins), weight_name=name)
            self.members[f.name] = tuple(lins)
            fused.append(f)
        self.linears: Tuple[LinearCase, ...] = tuple(fused)
        self.description = work.description + " (linears sharing an input fused along N)"

    def activation(self, lin: LinearCase, rows: int | None = None) -> np.ndarray:
        return self.base.activation(self.members[lin.name][0], rows=rows)

    def weight(self, lin: LinearCase) -> np.ndarray:
        return np.concatenate([self.base.weight(l) for l in self.members[lin.name]], axis=1)

    def grad(self, lin: LinearCase, rows: int | None = None) -> np.ndarray:
        return np.concatenate([self.base.grad(l, rows=rows) for l in self.members[lin.name]], axis=1)


def fuse_shared_inputs(work: Workload) -> FusedWorkload:
    return FusedWorkload(work)
