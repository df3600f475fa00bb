"""MoE FFN layer oracle (test infrastructure only).

Top-k softmax router, SwiGLU experts and a combine summed in fixed slot order.
Every token is evaluated directly against its own selected experts: there is no
permutation, no padding, no capacity and no layout at all, which is the result
both of the article's layouts must reach ([Article] §4.4, "Expert GEMM: two
layouts, same row result"; §4.5, "accumulated in FP32 in top-k slot order").

Readings where the pages are silent:
  * Router: the top-k is chosen by logit, descending, ties to the lower expert
    id; slot 0 holds the best expert.  The weights are the softmax over the k
    selected logits (equal, in exact arithmetic, to renormalising the full
    softmax over the selected experts), computed in fp32 in slot order.
  * No shared expert, no capacity drop, no router bias.
  * Each expert output is rounded to bf16 before the combine; the combine sums
    w[t, s] * y[t, s] in fp32 for s = 0 .. k-1 in that order and rounds once.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own.
"""
from __future__ import annotations

import numpy as np

from . import ops
from .bf16 import round_bf16

F32 = np.float32


def route_topk(logits, k: int):
    """Select k experts per token and their weights.

    [Article] §2 "the same discrete choices" (fixed tie-break and order) and
    §4.4 (one fp32 router output at every batch size).
    Returns ids int32 [T, k] (slot order) and weights fp32 [T, k].
    """
    x = np.asarray(logits, dtype=F32)
    T, E = x.shape
    # stable sort on -logit keeps equal logits in ascending expert-id order
    order = np.argsort(-x, axis=1, kind="stable")[:, :k].astype(np.int32)
    sel = np.take_along_axis(x, order, axis=1)
    e = np.exp(sel - sel[:, :1]).astype(F32)
    den = np.zeros((T, 1), dtype=F32)
    for s in range(k):  # slot-order sum
        den = den + e[:, s: s + 1]
    return order, (e / den).astype(F32)


def expert_ffn(x, w13, w2):
    """One SwiGLU expert on rows x: bf16(bf16(silu(g)*u) W2^T), g/u = bf16(x W13^T) halves."""
    F = w2.shape[1]
    g = ops.linear(x, w13[:F])
    u = ops.linear(x, w13[F:])
    return ops.linear(ops.silu_mul(g, u), w2)


def expert_outputs(x, ids, w13, w2):
    """y[t, s] = expert_ffn(x[t]) for expert ids[t, s]; fp32 [T, k, d] holding bf16 values.

    Rows of one expert are stacked into one matrix product purely to save time;
    each output element is still its own fp32 dot product.
    """
    x = np.asarray(x, dtype=F32)
    T, k = ids.shape
    d = np.asarray(w2).shape[1]
    y = np.empty((T, k, d), dtype=F32)
    for e in np.unique(ids):
        tt, ss = np.nonzero(ids == e)
        y[tt, ss] = expert_ffn(x[tt], np.asarray(w13[e], dtype=F32), np.asarray(w2[e], dtype=F32))
    return y


def combine(y, weights):
    """out[t] = bf16( sum_{s=0..k-1} w[t, s] * y[t, s] ), fp32, sequential slot order."""
    y = np.asarray(y, dtype=F32)
    w = np.asarray(weights, dtype=F32)
    acc = np.zeros((y.shape[0], y.shape[2]), dtype=F32)
    for s in range(y.shape[1]):
        acc = acc + w[:, s: s + 1] * y[:, s, :]
    return round_bf16(acc)


def moe_layer(x, router_logits, w13, w2, k: int):
    """Full MoE FFN: route, run the selected experts per token, combine in slot order."""
    ids, wts = route_topk(router_logits, k)
    y = expert_outputs(x, ids, w13, w2)
    return combine(y, wts), ids, wts
