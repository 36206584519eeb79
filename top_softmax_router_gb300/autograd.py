"""torch.autograd wrappers over the C ABI: the MoE block and the vocabulary cross-entropy head as
differentiable functions, so they drop into a training loop.

Argument marshalling only: forward and backward call the library's moe_route / moe_forward /
moe_backward and moe_ce_forward / moe_ce_backward.  The library returns fp32 weight gradients;
autograd hands each gradient back in its parameter's dtype, so bf16 weights receive bf16
gradients.  (A caller that keeps fp32 master weights and wants the fp32 gradients uses MoEBlock /
VocabCE directly.)
"""
from __future__ import annotations

import torch

from .api import MoEBlock
from .ce import VocabCE

__all__ = ["MoEFunction", "VocabCEFunction", "moe_block", "vocab_cross_entropy"]


class MoEFunction(torch.autograd.Function):
    """Y = MoE(X) with top-k softmax routing (Wr, bias), SwiGLU experts (Wg, Wu, Wd), chunked by (c, K_max).
    Gradients flow to X, Wr, Wg, Wu and Wd; the bias gets none (it only shifts the routing)."""

    @staticmethod
    def forward(ctx, X, Wr, bias, Wg, Wu, Wd, blk: MoEBlock):
        idx, gates = blk.route(X, Wr, bias)
        Y = blk.forward(X, idx, gates, Wg, Wu, Wd)
        ctx.blk = blk
        ctx.save_for_backward(X, Wr, Wg, Wu, Wd, idx, gates)
        return Y

    @staticmethod
    def backward(ctx, dY):
        X, Wr, Wg, Wu, Wd, idx, gates = ctx.saved_tensors
        g = ctx.blk.backward(X, Wr, idx, gates, Wg, Wu, Wd, dY.contiguous(), want_dgates=False)
        return g["dX"], g["dWr"], None, g["dWg"], g["dWu"], g["dWd"], None


def moe_block(X, Wr, bias, Wg, Wu, Wd, blk: MoEBlock):
    """Differentiable MoE block over an MoEBlock's workspace (X [N,H] bf16; weights as in include/moe.h)."""
    return MoEFunction.apply(X, Wr, bias, Wg, Wu, Wd, blk)


class VocabCEFunction(torch.autograd.Function):
    """Mean cross-entropy of the logits X W^T against `targets`, without forming the logits."""

    @staticmethod
    def forward(ctx, X, W, targets, ce: VocabCE):
        loss, lse, mean = ce.forward(X, W, targets)
        ctx.ce = ce
        ctx.save_for_backward(X, W, targets, lse)
        return mean[0]

    @staticmethod
    def backward(ctx, dmean):
        X, W, targets, lse = ctx.saved_tensors
        n = X.shape[0]
        dloss = (dmean.float() / max(n, 1)).expand(n).contiguous()
        dX, dW = ctx.ce.backward(X, W, targets, lse, dloss)
        return dX, dW, None, None


def vocab_cross_entropy(X, W, targets, ce: VocabCE):
    """Differentiable mean cross-entropy head over a VocabCE's workspace."""
    return VocabCEFunction.apply(X, W, targets, ce)
