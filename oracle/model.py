"""Whole-decoder oracle (test infrastructure only).

A pre-norm decoder with RoPE, causal GQA attention and a SwiGLU FFN, ending in
fp32 logits and the sampled token's logprob.  The residual stream is carried in
bf16 and every sub-layer output is rounded to bf16 once, as in ``ops``.  The
oracle runs one sequence at a time over its whole prefix, so it has no batch,
no chunking, no paging and no KV split at all: the article's requirement is
that the GPU results reach the same values whatever those are ([Article] §2:
batch independence, phase consistency).

Layer (pre-norm):
    x  = rmsnorm(r, attn_norm)                  (first layer: r = embed[ids])
    q,k,v = split(bf16(x Wqkv^T));  q,k = rope(q), rope(k)
    a  = attention(q, k, v)
    r, x = rmsnorm(bf16(x Wo^T) + r, ffn_norm)  (fused residual add)
    g,u = bf16(x Wg^T), bf16(x Wu^T);  y = silu_mul(g, u)
    r  = bf16(r + bf16(y W2^T))                 (added by the next norm)
Final: x = rmsnorm(r, final_norm); logits = x Wlm^T (fp32).

Weights are dicts of fp32 arrays holding bf16 values (see ``weights_to_f32``).

Block-FP8 model ("vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 W8A8
linear layers, §4.2 FP8 KV cache), weights from ``fp8_weights``: the four
linear layers of every block become W8A8 GEMMs (the bf16 input rows quantised
in 1 x 128 blocks, the weights in 128 x 128 blocks, bf16 output), and K (after
RoPE) and V make the FP8 round trip of the cache (one power-of-two scale per
token and kv head) before attention reads them.  Everything else, the lm_head
included, is the bf16 model unchanged (the lm_head staying bf16 is a reading:
the pages name the dense GEMMs of the blocks).
"""
from __future__ import annotations

import numpy as np

from . import fp8 as ofp8
from . import ops
from .bf16 import bf16_bits_to_f32, round_bf16

F32 = np.float32


def weights_to_f32(w_bits: dict) -> dict:
    """Convert a weight dict of bf16 bit arrays into exact fp32 arrays."""
    out = {k: bf16_bits_to_f32(w_bits[k]) for k in ("embed", "final_norm", "lm_head")}
    out["layers"] = [{k: bf16_bits_to_f32(v) for k, v in lw.items()} for lw in w_bits["layers"]]
    return out


FP8_LINEARS = ("wqkv", "wo", "w13", "w2")


def fp8_weights(w: dict) -> dict:
    """The block-FP8 model made from bf16 masters by the deployment rule
    ([Article] §4.1: training quantises its bf16 master weights to block FP8
    before the same GEMM): a copy of ``w`` whose layers also carry the codes
    and 128 x 128 block scales of the four linear weights under key "fp8"."""
    out = dict(w)
    out["layers"] = []
    for lw in w["layers"]:
        l8 = dict(lw)
        l8["fp8"] = {k: ofp8.quantize_weight(lw[k]) for k in FP8_LINEARS}
        out["layers"].append(l8)
    return out


def linear_fp8(x, qw, sw):
    """W8A8 linear layer: bf16 rows x quantised in 1 x 128 blocks, times the
    block-FP8 weight, rounded once to bf16 ([Article] §4.1)."""
    qa, sa = ofp8.quantize_act(x)
    return ofp8.gemm_fp8(qa, sa, qw, sw, out="bf16")


def kv_round_trip(t):
    """K or V [L, Hkv, hd] as attention reads them from the FP8 cache: each
    (token, kv head) vector quantised with its own power-of-two scale, then
    dequantised ([Article] §4.2)."""
    n, h, hd = t.shape
    q, s = ofp8.quantize_blocks(np.asarray(t, F32).reshape(n * h, hd), 1, block_cols=hd)
    return ofp8.dequantize_blocks(q, s, 1, block_cols=hd).reshape(n, h, hd)


def layer(lw: dict, shape, r, pos, return_parts: bool = False):
    """One decoder layer on the residual stream r [L, d] of ONE sequence whose
    rows sit at positions ``pos`` (0 .. L-1, every earlier key is in r).
    Returns the residual stream after the layer, bf16(r + attn + ffn) with the
    two adds rounded separately (and, with ``return_parts``, the attention
    output projection o and the FFN output dn that were added)."""
    L = r.shape[0]
    hq, hkv, hd, F = shape.n_heads_q, shape.n_heads_kv, shape.head_dim, shape.ffn
    w8 = lw.get("fp8")
    x, _ = ops.rmsnorm(r, lw["attn_norm"], shape.eps)
    qkv = linear_fp8(x, *w8["wqkv"]) if w8 else ops.linear(x, lw["wqkv"])
    q = qkv[:, : hq * hd].reshape(L, hq, hd)
    k = qkv[:, hq * hd: (hq + hkv) * hd].reshape(L, hkv, hd)
    v = qkv[:, (hq + hkv) * hd:].reshape(L, hkv, hd)
    q = ops.rope(q, pos, shape.rope_theta)
    k = ops.rope(k, pos, shape.rope_theta)
    if w8:
        k, v = kv_round_trip(k), kv_round_trip(v)
    a = ops.attention(q, k, v, pos).reshape(L, hq * hd)
    o = linear_fp8(a, *w8["wo"]) if w8 else ops.linear(a, lw["wo"])
    x, r = ops.rmsnorm(o, lw["ffn_norm"], shape.eps, residual=r)
    if w8:
        g13 = linear_fp8(x, *w8["w13"])
        g, u = g13[:, :F], g13[:, F:]
        dn = linear_fp8(ops.silu_mul(g, u), *w8["w2"])
    else:
        g = ops.linear(x, lw["w13"][:F])
        u = ops.linear(x, lw["w13"][F:])
        dn = ops.linear(ops.silu_mul(g, u), lw["w2"])
    out = round_bf16(r + dn)
    return (out, o, dn) if return_parts else out


def hidden_states(w: dict, shape, tokens, return_layers: bool = False):
    """Final-norm output for every position of one sequence, fp32 [L, d] (bf16 values).

    ``shape`` carries n_heads_q, n_heads_kv, head_dim, ffn, eps, rope_theta.
    With ``return_layers`` also returns the residual stream entering every
    layer and leaving the last one (n_layers + 1 arrays).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    pos = np.arange(tokens.shape[0])
    r = w["embed"][tokens]
    per_layer = [r]
    for lw in w["layers"]:
        r = layer(lw, shape, r, pos)
        per_layer.append(r)
    x, _ = ops.rmsnorm(r, w["final_norm"], shape.eps)
    if return_layers:
        return x, per_layer
    return x


def score(w: dict, shape, tokens, rows, targets):
    """Teacher-forced scoring of one sequence.

    Runs the forward over ``tokens`` and returns, for each row index in
    ``rows``, the fp32 logits row and the logprob (fp64) of ``targets`` at that
    row.  This is the training-side recomputation of [Article] §2 ("the training
    side's recomputed old-logprob") written as a plain definition.
    """
    x = hidden_states(w, shape, tokens)
    rows = np.asarray(rows, dtype=np.int64)
    logits = ops.linear(x[rows], w["lm_head"], out="fp32")
    return logits, ops.logprob(logits, targets)


def score_generation(w: dict, shape, prompt, generated):
    """Logprobs of each generated token given the prompt and the earlier generated tokens.

    Generated token j (0-based) is predicted by the row at position
    len(prompt) + j - 1, so the forward runs over prompt + generated[:-1].
    Returns (logits [G, V] fp32, logprob [G] fp64, greedy argmax [G]).
    """
    prompt = np.asarray(prompt, dtype=np.int64)
    generated = np.asarray(generated, dtype=np.int64)
    seq = np.concatenate([prompt, generated[:-1]])
    rows = np.arange(len(prompt) - 1, len(seq))
    logits, lp = score(w, shape, seq, rows, generated)
    return logits, lp, ops.argmax_lowest(logits)


def greedy_generate(w: dict, shape, prompt, n_new: int):
    """Greedy decoding by repeated full-prefix recomputation (slow; tiny models only).

    Each step recomputes the whole prefix, so the oracle's decode is its
    prefill by construction.  Returns (generated ids [n_new], logprobs [n_new]).
    """
    seq = list(np.asarray(prompt, dtype=np.int64))
    ids, lps = [], []
    for _ in range(n_new):
        x = hidden_states(w, shape, np.asarray(seq))
        logits = ops.linear(x[-1:], w["lm_head"], out="fp32")
        t = int(ops.argmax_lowest(logits)[0])
        ids.append(t)
        lps.append(float(ops.logprob(logits, [t])[0]))
        seq.append(t)
    return np.asarray(ids, dtype=np.int32), np.asarray(lps)


def logprob_head(h, gain, lm_head, ids, eps: float = 1e-6, norm: bool = True):
    """Logprob head alone: optional RMSNorm, fp32-output lm_head GEMM, log-softmax + gather.

    Returns (logits fp32 [T, V], logprob fp64 [T]).
    """
    x = ops.rmsnorm(h, gain, eps)[0] if norm else np.asarray(h, dtype=F32)
    logits = ops.linear(x, lm_head, out="fp32")
    return logits, ops.logprob(logits, ids)
