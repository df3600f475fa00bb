"""Per-operator definitions of the decoder forward (oracle; test infrastructure only).

Each function is the plain definition of one step of the hot path, written in
numpy with fp32 accumulation and bf16 rounding (round-to-nearest-even) at the
layer boundary that the GPU path also rounds at.  All bf16 tensors are carried
as fp32 arrays whose values are exactly bf16-representable.

Readings of the pages where they leave a step open (each is the plainest
reading the rest supports):
  * RMSNorm epsilon 1e-6; y = x * (1 / sqrt(mean(x^2) + eps)) * g.
  * RoPE: rotate-half pairs (i, i + hd/2), angle pos * theta^(-2i/hd), base 10000,
    cos/sin evaluated in fp64 and rounded to fp32, applied in fp32, rounded to bf16.
  * Attention: causal, scale 1/sqrt(hd), query head h reads kv head
    h // (Hq / Hkv); explicit softmax over all keys j <= position.
  * Logits are kept fp32; the logprob is logit[id] - logsumexp(logits), the
    logsumexp taken in fp64.
  * Greedy choice: argmax with ties going to the lowest token id.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_bf16

F32 = np.float32


def rmsnorm(x, gain, eps: float = 1e-6, residual=None):
    """RMSNorm with an optional residual add in front of it.

    [Article] §3.1 names RMSNorm among the small operators whose forward values
    come from the inference kernel; §2 "batch independence" requires the row
    result to depend on the row only, which this per-row definition does.

    If ``residual`` is given: r = bf16(residual + x) (the residual stream is
    carried in bf16), else r = x.  Then
        y = bf16( r * (1 / sqrt(sum(r^2) / d + eps)) * g )   (fp32 arithmetic)
    Returns (y, r).
    """
    x = np.asarray(x, dtype=F32)
    if residual is not None:
        r = round_bf16(np.asarray(residual, dtype=F32) + x)
    else:
        r = x
    d = r.shape[-1]
    ms = np.sum(r * r, axis=-1, dtype=F32, keepdims=True) / F32(d)
    inv = F32(1.0) / np.sqrt(ms + F32(eps), dtype=F32)
    y = round_bf16((r * inv) * np.asarray(gain, dtype=F32))
    return y, r


def linear(x, w, out: str = "bf16"):
    """Dense GEMM C[m, n] = sum_k A[m, k] * W[n, k], fp32 accumulation.

    [Article] §4.1 "Dense GEMM: one accumulation order for every M": the value
    of a row may not depend on M.  The definition below has no M dependence at
    all.  ``out='bf16'`` rounds the result once to bf16; ``out='fp32'`` keeps it
    (the router gate and the lm_head keep fp32 outputs, §4.1 / §4.4).
    """
    a = np.asarray(x, dtype=F32)
    b = np.asarray(w, dtype=F32)
    c = np.matmul(a, b.T).astype(F32)
    if out == "bf16":
        return round_bf16(c)
    if out == "fp32":
        return c
    raise ValueError(out)


def rope_cos_sin(positions, head_dim: int, theta: float = 10000.0):
    """cos/sin of pos * theta^(-2i/hd) for i < hd/2, computed in fp64, rounded to fp32."""
    pos = np.asarray(positions, dtype=np.float64)
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * i / head_dim)
    ang = pos[:, None] * inv_freq[None, :]
    return np.cos(ang).astype(F32), np.sin(ang).astype(F32)


def rope(x, positions, theta: float = 10000.0):
    """Rotate-half rotary embedding of x [T, H, hd] at absolute positions [T].

    out[i]        = bf16( x[i] * cos - x[i + hd/2] * sin )
    out[i + hd/2] = bf16( x[i + hd/2] * cos + x[i] * sin )
    The position is the token's absolute position within its own sequence, so
    the result never depends on batch-mates ([Article] §2, batch independence;
    §4.3 makes the same point for the in-request position).
    """
    x = np.asarray(x, dtype=F32)
    hd = x.shape[-1]
    c, s = rope_cos_sin(positions, hd, theta)
    c = c[:, None, :]
    s = s[:, None, :]
    x1 = x[..., : hd // 2]
    x2 = x[..., hd // 2:]
    o1 = x1 * c - x2 * s
    o2 = x2 * c + x1 * s
    return round_bf16(np.concatenate([o1, o2], axis=-1))


def attention(q, k, v, q_pos, k_len=None, row_block: int = 256):
    """Causal GQA attention with an explicit softmax (no splits, no tiles).

    q [Tq, Hq, hd] at absolute positions q_pos [Tq]; k, v [Tk, Hkv, hd] hold the
    keys/values of positions 0..Tk-1 of the same sequence.  Row i attends to
    keys j <= q_pos[i]:
        s_j = (q_i . k_j) / sqrt(hd)       (fp32)
        P_j = exp(s_j - max_j s_j) / sum_j exp(s_j - max_j s_j)
        o_i = bf16( sum_j P_j v_j )
    [Article] §4.2: prefill, decode and training must read the history through
    one algorithm; the result they must all reach is this definition.  Rows are
    processed in blocks only to bound memory; each row's softmax is complete.
    """
    q = np.asarray(q, dtype=F32)
    k = np.asarray(k, dtype=F32)
    v = np.asarray(v, dtype=F32)
    q_pos = np.asarray(q_pos, dtype=np.int64)
    tq, hq, hd = q.shape
    hkv = k.shape[1]
    group = hq // hkv
    scale = F32(1.0) / np.sqrt(F32(hd), dtype=F32)
    out = np.empty((tq, hq, hd), dtype=F32)
    kpos = np.arange(k.shape[0])
    for h in range(hq):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        for r0 in range(0, tq, row_block):
            r1 = min(tq, r0 + row_block)
            s = np.matmul(q[r0:r1, h, :], kh.T).astype(F32) * scale
            mask = kpos[None, :] <= q_pos[r0:r1, None]
            s = np.where(mask, s, F32(-np.inf))
            m = np.max(s, axis=1, keepdims=True)
            p = np.exp(s - m).astype(F32)
            p = np.where(mask, p, F32(0.0))
            den = np.sum(p, axis=1, keepdims=True, dtype=F32)
            o = np.matmul(p / den, vh).astype(F32)
            out[r0:r1, h, :] = o
    return round_bf16(out)


def silu_mul(gate, up):
    """SwiGLU activation a = bf16( silu(g) * u ), silu(g) = g / (1 + exp(-g)).

    [Article] §4.4, condition 3: SiLU(gate) x up is computed in fp32 and only
    the product is rounded (once) to bf16.
    """
    g = np.asarray(gate, dtype=F32)
    u = np.asarray(up, dtype=F32)
    with np.errstate(over="ignore"):
        silu = g / (F32(1.0) + np.exp(-g).astype(F32))
    return round_bf16(silu * u)


def logprob(logits, ids):
    """Log-probability of the sampled id: x[id] - logsumexp(x), logsumexp in fp64.

    [Article] §2: diff is defined on the logprob of each sampled token; §3.1
    lists "the final logprob" as a fused output of the forward.
    Returns fp64 [T].
    """
    x = np.asarray(logits, dtype=np.float64)
    ids = np.asarray(ids, dtype=np.int64)
    m = np.max(x, axis=-1, keepdims=True)
    lse = m[..., 0] + np.log(np.sum(np.exp(x - m), axis=-1))
    return x[np.arange(x.shape[0]), ids] - lse


def argmax_lowest(logits):
    """Greedy choice: argmax over the vocab, ties to the lowest id.

    [Article] §2 "the same discrete choices": tie-breaking must be fixed.
    (numpy's argmax returns the first maximal index.)
    """
    return np.argmax(np.asarray(logits, dtype=F32), axis=-1).astype(np.int32)


def diff_stats(lp_rollout, lp_train):
    """Acceptance statistics of [Article] §2 and §3.2.

    diff_t = |lp_rollout_t - lp_train_t|; returns max, mean and (population)
    std of diff, and the k3 KL estimator mean(r - 1 - log r) with
    r = exp(lp_train - lp_rollout), all in fp64.  All four are exactly 0 iff the
    two logprob vectors are identical.
    """
    a = np.asarray(lp_rollout, dtype=np.float64)
    b = np.asarray(lp_train, dtype=np.float64)
    d = np.abs(a - b)
    logr = b - a
    k3 = np.expm1(logr) - logr
    if d.size == 0:
        return {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}
    return {"max": float(d.max()), "mean": float(d.mean()), "std": float(d.std()),
            "k3": float(k3.mean())}
