"""Noise floor of the free-running logprob tolerance (test infrastructure, CPU only).

The GPU path and the oracle implement one numerical contract (fp32 accumulation,
bf16 rounding at the same layer boundaries) but sum in different orders, and the
attention kernel rounds the probabilities P to bf16 before P.V where the oracle
keeps them in fp32.  Two legitimate implementations of the contract therefore
differ by one-ulp bf16 flips in the residual stream, and those flips propagate
through the later layers to the logprobs.  How far apart they drift depends on the
model, so the free-running tolerance is measured here, per model, as the distance
between the oracle and variants of itself that make exactly those two changes:

  * ``fp64``:   every GEMM and the attention accumulated in fp64 (then rounded at
    the same boundaries as before);
  * ``bf16p``:  attention as an online softmax over 64-key tiles in ascending
    order, fp32 running max and sum, P rounded to bf16 before P.V (the sum of P
    stays fp32), which is what the kernel does per row;
  * ``both``:   the two changes together.

The variants replace ``oracle.ops.linear`` and ``oracle.ops.attention`` for the
duration of one scoring call; ``oracle.model`` reaches both through the module.
Scoring is teacher forced on seeded uniform continuation tokens (on the CPU there
are no GPU-sampled ids; the model's arithmetic does not depend on which ids were
chosen).
"""
from __future__ import annotations

import contextlib

import numpy as np

from oracle import model as omodel
from oracle import ops
from oracle.bf16 import round_bf16

F32 = np.float32


def linear_fp64(x, w, out: str = "bf16"):
    """C = A W^T accumulated in fp64, then rounded as the oracle rounds its fp32 result."""
    c = np.matmul(np.asarray(x, np.float64), np.asarray(w, np.float64).T)
    if out == "bf16":
        return round_bf16(c.astype(F32))
    if out == "fp32":
        return c.astype(F32)
    raise ValueError(out)


def attention_fp64(q, k, v, q_pos, k_len=None, row_block: int = 256):
    """Causal GQA attention with an explicit softmax, all in fp64, output rounded to bf16."""
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    q_pos = np.asarray(q_pos, np.int64)
    tq, hq, hd = q.shape
    group = hq // k.shape[1]
    out = np.empty((tq, hq, hd), np.float64)
    kpos = np.arange(k.shape[0])
    for h in range(hq):
        kh, vh = k[:, h // group, :], v[:, h // group, :]
        for r0 in range(0, tq, row_block):
            r1 = min(tq, r0 + row_block)
            s = (q[r0:r1, h, :] @ kh.T) / np.sqrt(hd)
            mask = kpos[None, :] <= q_pos[r0:r1, None]
            s = np.where(mask, s, -np.inf)
            p = np.where(mask, np.exp(s - s.max(axis=1, keepdims=True)), 0.0)
            out[r0:r1, h, :] = (p / p.sum(axis=1, keepdims=True)) @ vh
    return round_bf16(out.astype(F32))


def _attention_online(q, k, v, q_pos, acc_dtype, row_block: int = 256, tile: int = 64):
    """Online softmax over `tile`-key tiles in ascending order: running max m and
    sum l in fp32, P = exp(s - m) rounded to bf16 for P.V (l sums the unrounded P),
    P.V and the rescaled accumulator in `acc_dtype`; out = bf16(acc / l)."""
    q = np.asarray(q, F32)
    k = np.asarray(k, F32)
    v = np.asarray(v, F32)
    q_pos = np.asarray(q_pos, np.int64)
    tq, hq, hd = q.shape
    group = hq // k.shape[1]
    scale = F32(1.0) / np.sqrt(F32(hd), dtype=F32)
    out = np.empty((tq, hq, hd), F32)
    n_keys = int(q_pos.max()) + 1
    for h in range(hq):
        kh, vh = k[:, h // group, :], v[:, h // group, :]
        for r0 in range(0, tq, row_block):
            r1 = min(tq, r0 + row_block)
            qs = q[r0:r1, h, :]
            pos = q_pos[r0:r1, None]
            m = np.full((r1 - r0, 1), -np.inf, F32)
            l = np.zeros((r1 - r0, 1), F32)
            acc = np.zeros((r1 - r0, hd), acc_dtype)
            for k0 in range(0, n_keys, tile):
                k1 = min(n_keys, k0 + tile)
                kp = np.arange(k0, k1)[None, :]
                ok = kp <= pos
                if not ok.any():
                    break
                s = np.matmul(qs.astype(acc_dtype), kh[k0:k1].T.astype(acc_dtype)).astype(F32) * scale
                s = np.where(ok, s, F32(-np.inf))
                m_new = np.maximum(m, s.max(axis=1, keepdims=True))
                with np.errstate(invalid="ignore"):
                    alpha = np.where(m_new == m, F32(1.0), np.exp(m - m_new).astype(F32))
                p = np.where(ok, np.exp(s - m_new).astype(F32), F32(0.0))
                l = l * alpha + p.sum(axis=1, keepdims=True, dtype=F32)
                acc = acc * alpha.astype(acc_dtype) + np.matmul(round_bf16(p).astype(acc_dtype),
                                                                vh[k0:k1].astype(acc_dtype))
                m = m_new
            out[r0:r1, h, :] = (acc / l.astype(acc_dtype)).astype(F32)
    return round_bf16(out)


def attention_bf16p(q, k, v, q_pos, k_len=None, row_block: int = 256):
    return _attention_online(q, k, v, q_pos, F32, row_block)


def attention_both(q, k, v, q_pos, k_len=None, row_block: int = 256):
    return _attention_online(q, k, v, q_pos, np.float64, row_block)


VARIANTS = {
    "fp64": (linear_fp64, attention_fp64),
    "bf16p": (None, attention_bf16p),
    "both": (linear_fp64, attention_both),
}


@contextlib.contextmanager
def variant(name: str):
    """Swap oracle.ops.linear / oracle.ops.attention for the named variant."""
    lin, att = VARIANTS[name]
    saved = ops.linear, ops.attention
    try:
        if lin is not None:
            ops.linear = lin
        ops.attention = att
        yield
    finally:
        ops.linear, ops.attention = saved


def floors(W, shape, prompts, gens, names=("fp64", "bf16p", "both")):
    """Teacher-forced logprobs of `gens` after `prompts` from the oracle and from each
    variant; returns {variant: (max, mean, p99) of |variant - oracle|} over all tokens."""
    base = np.concatenate([omodel.score_generation(W, shape, p, g)[1] for p, g in zip(prompts, gens)])
    res = {}
    for name in names:
        with variant(name):
            lp = np.concatenate([omodel.score_generation(W, shape, p, g)[1] for p, g in zip(prompts, gens)])
        e = np.abs(lp - base)
        res[name] = (float(e.max()), float(e.mean()), float(np.quantile(e, 0.99)))
    return res
