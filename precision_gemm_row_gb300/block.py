"""One LLaMA decoder block trained on synthetic tokens, with its seven linear
layers on the FP4 library.

The pages (page "首个 FP4 精度的大模型训练框架来了", czzqal.com, and page
"Optimizing Large Language Model Training Using FP4 Quantization", abstract)
train LLaMA models whose linear layers run the quantized path: FP4 forward
with outlier clamping and compensation, and a backward whose weight gradient
carries the DGE correction.  Here one block is stepped end to end to exercise
that loop: every q/k/v/o and gate/up/down product goes through
fp4lin.linear_forward (quantile clamp + CSR, row and column E2M1
quantization, FP4 GEMM with compensation) and fp4lin.linear_backward (DGE
weight gradient, input gradient); the non-GEMM parts (RMSNorm, rotary
embedding, attention softmax, SiLU, residuals) are plain BF16 torch ops, which
the pages leave in higher precision.  The loss is a stand-in (a squared error
against a seeded target) and the update plain SGD on fp32 master weights; no
dataset, no claim about accuracy.  With fp8_grads the weight gradients leave
the GEMM as E4M3 codes with a per-tensor scale set from the previous step's
max |dW| (the page's FP8 gradient communication; the first step, with no
history, uses fp32), and the update uses their dequantized values.

Every linear runs on the CUDA library: without it (or without a GPU) the
calls fail loudly, there is no fallback.
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Dict, List, Optional

import torch
import torch.nn.functional as F

from . import fp4lin

LINEARS = ("q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj")


@dataclass
class BlockConfig:
    hidden: int = 1024
    heads: int = 8
    ffn: int = 2816
    batch: int = 2
    seq: int = 1024
    vocab: int = 4096
    q: float = 0.999           # quantile of |A| clamped in every activation
    dge_k: float = 5.0
    dge_clip: float = 3.0
    lr: float = 0.1
    loss_scale: float = 1.0    # static loss scale (the gradients are unscaled before the update)
    fp8_grads: bool = False    # weight gradients as E4M3 codes (delayed per-tensor scale), as communicated
    seed: int = 0


class _FP4Linear(torch.autograd.Function):
    """Y = A W on the FP4 path; backward = (dY W^T, DGE-corrected A^T dY)."""

    @staticmethod
    def forward(ctx, A: torch.Tensor, W_master: torch.Tensor, cfg: BlockConfig, name: str,
                record: Optional[Dict[str, dict]], amax: Optional[Dict[str, torch.Tensor]] = None):
        A = A.contiguous()
        W = W_master.to(torch.bfloat16)
        Y, inter = fp4lin.linear_forward(A, W, cfg.q)
        ctx.save_for_backward(A, W, inter["s_w"])
        ctx.cfg, ctx.name, ctx.record, ctx.amax = cfg, name, record, amax
        if record is not None:
            record[name] = dict(A=A, W=W, s_w=inter["s_w"], nnz=int(inter["outlier"]["nnz"].item()))
        return Y

    @staticmethod
    def backward(ctx, dY: torch.Tensor):
        A, W, s_w = ctx.saved_tensors
        cfg = ctx.cfg
        dY = dY.to(torch.bfloat16).contiguous()
        dX = fp4lin.fp4_linear_dgrad(dY, W)
        prev = ctx.amax.get(ctx.name) if (cfg.fp8_grads and ctx.amax is not None) else None
        if prev is None:
            dW = fp4lin.fp4_linear_wgrad_dge(A, dY, W, s_w, cfg.dge_k, cfg.dge_clip)
            if cfg.fp8_grads and ctx.amax is not None:
                ctx.amax[ctx.name] = dW.abs().amax().reshape(1)
        else:
            # delayed scaling: the previous step's max |dW| sets this step's scale
            scale = (448.0 / torch.clamp(prev, min=1e-30)).to(torch.float32)
            codes, amax = fp4lin.fp4_linear_wgrad_dge(A, dY, W, s_w, cfg.dge_k, cfg.dge_clip, dw_type="e4m3",
                                                     dw_scale=scale)
            ctx.amax[ctx.name] = amax
            dW = codes.view(torch.float8_e4m3fn).to(torch.float32) / scale
        if ctx.record is not None:
            ctx.record[ctx.name].update(dY=dY, dW=dW)
        return dX, dW, None, None, None, None


def _rms_norm(x: torch.Tensor, eps: float = 1e-6) -> torch.Tensor:
    xf = x.float()
    return (xf * torch.rsqrt(xf.pow(2).mean(-1, keepdim=True) + eps)).to(x.dtype)


def _rope(x: torch.Tensor) -> torch.Tensor:
    """Rotary position embedding over (batch, heads, seq, head_dim), base 10000."""
    S, D = x.shape[-2], x.shape[-1]
    inv = 1.0 / (10000.0 ** (torch.arange(0, D, 2, device=x.device, dtype=torch.float32) / D))
    ang = torch.arange(S, device=x.device, dtype=torch.float32)[:, None] * inv[None, :]
    cos, sin = ang.cos(), ang.sin()
    x1, x2 = x.float()[..., 0::2], x.float()[..., 1::2]
    out = torch.stack((x1 * cos - x2 * sin, x1 * sin + x2 * cos), dim=-1).flatten(-2)
    return out.to(x.dtype)


class LlamaBlock:
    """Pre-norm LLaMA block: h = x + Attn(RMSNorm(x)); y = h + MLP(RMSNorm(h)),
    MLP = down(SiLU(gate(.)) * up(.)), causal multi-head attention with rotary
    embeddings.  Weights are K x N (in x out) fp32 masters, N(0, 0.02)."""

    def __init__(self, cfg: BlockConfig, device="cuda"):
        if cfg.hidden % cfg.heads:
            raise ValueError("hidden must be a multiple of heads")
        self.cfg = cfg
        g = torch.Generator(device="cpu").manual_seed(cfg.seed)
        shapes = dict(q_proj=(cfg.hidden, cfg.hidden), k_proj=(cfg.hidden, cfg.hidden),
                      v_proj=(cfg.hidden, cfg.hidden), o_proj=(cfg.hidden, cfg.hidden),
                      gate_proj=(cfg.hidden, cfg.ffn), up_proj=(cfg.hidden, cfg.ffn),
                      down_proj=(cfg.ffn, cfg.hidden))
        self.W = {n: (torch.randn(shapes[n], generator=g) * 0.02).to(device).requires_grad_(True)
                  for n in LINEARS}
        self.embed = (torch.randn((cfg.vocab, cfg.hidden), generator=g)).to(device, torch.bfloat16)
        tokens = torch.randint(0, cfg.vocab, (cfg.batch, cfg.seq), generator=g)
        self.tokens = tokens.to(device)
        self.target = (torch.randn((cfg.batch * cfg.seq, cfg.hidden), generator=g)).to(device, torch.bfloat16)
        self.amax: Dict[str, torch.Tensor] = {}   # per linear: last step's max |dW| (FP8 gradients)

    def _lin(self, x: torch.Tensor, name: str, record) -> torch.Tensor:
        return _FP4Linear.apply(x, self.W[name], self.cfg, name, record, self.amax)

    def forward(self, record: Optional[Dict[str, dict]] = None) -> torch.Tensor:
        c = self.cfg
        M, D = c.batch * c.seq, c.hidden // c.heads
        x = self.embed[self.tokens.reshape(-1)]                                  # (M, hidden) bf16
        xn = _rms_norm(x)
        q, k, v = (self._lin(xn, n, record) for n in ("q_proj", "k_proj", "v_proj"))
        split = lambda t: t.view(c.batch, c.seq, c.heads, D).transpose(1, 2)
        att = F.scaled_dot_product_attention(_rope(split(q)), _rope(split(k)), split(v), is_causal=True)
        att = att.transpose(1, 2).reshape(M, c.hidden)
        h = x + self._lin(att, "o_proj", record)
        hn = _rms_norm(h)
        mlp = F.silu(self._lin(hn, "gate_proj", record)) * self._lin(hn, "up_proj", record)
        y = h + self._lin(mlp, "down_proj", record)
        return y

    def loss(self, y: torch.Tensor) -> torch.Tensor:
        """Stand-in loss: half the squared error to the seeded target, per token."""
        d = y.float() - self.target.float()
        return 0.5 * d.pow(2).sum() / d.shape[0]

    def step(self, record: Optional[Dict[str, dict]] = None) -> float:
        """One training step: forward, loss, backward through the library's
        DGE weight gradient and input gradient, SGD update.  Returns the loss."""
        for w in self.W.values():
            w.grad = None
        loss = self.loss(self.forward(record))
        (loss * self.cfg.loss_scale).backward()
        with torch.no_grad():
            for w in self.W.values():
                w.add_(w.grad, alpha=-self.cfg.lr / self.cfg.loss_scale)
        return float(loss.item())


def train(cfg: BlockConfig, steps: int, device="cuda") -> List[float]:
    """Losses of `steps` SGD steps of one block on its synthetic tokens."""
    block = LlamaBlock(cfg, device)
    return [block.step() for _ in range(steps)]
