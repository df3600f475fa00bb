"""Seeded synthetic workloads for the batch-invariant decoder forward.

Every tensor is drawn from ``numpy.random.default_rng(seed)`` in a fixed order,
so both sides of every comparison see the same bits.  bf16 tensors are returned
as ``uint16`` arrays holding the bf16 bit pattern.  Nothing here computes any
part of the forward; the shapes and distributions follow the workloads that the
batch-invariance article describes (dense decoder, MoE layer, large-vocab
logprob head, long-context GQA decoder).
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

__all__ = [
    "DecoderShape", "C1", "C2", "C3", "C4", "C5",
    "to_bf16_bits", "bits_to_f32", "normal_bf16",
    "make_decoder_weights", "make_prompts", "make_logprob_head", "make_moe_layer",
    "make_c5_prompt_lengths",
]


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 array -> bf16 bit patterns (uint16), converted by torch on the CPU."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) -> the fp32 values they represent (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float) -> np.ndarray:
    """N(0, std^2) samples rounded to bf16, as uint16 bits."""
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return to_bf16_bits(x)


@dataclasses.dataclass(frozen=True)
class DecoderShape:
    n_layers: int
    d: int
    n_heads_q: int
    n_heads_kv: int
    head_dim: int
    ffn: int
    vocab: int
    eps: float = 1e-6
    rope_theta: float = 10000.0
    kv_block: int = 64
    kv_split: int = 512


# The five workloads.
C1 = dict(n_seq=8, seq_len=64, d=256, vocab=4096, w_std=0.02, seed=101)
C2 = dict(shape=DecoderShape(4, 512, 8, 8, 64, 1408, 32000), w_std=0.02, batch=16,
          prompt_min=128, prompt_max=512, gen=256, seed=202)
C3 = dict(n_tokens=4096, d=2048, ffn=1024, n_experts=64, top_k=8, w_std=0.02, seed=303)
C4 = dict(n_tokens=16384, d=4096, vocab=129280, w_std=0.01, seed=404)
C5 = dict(shape=DecoderShape(8, 2048, 16, 4, 128, 5632, 32000), w_std=0.02, batch=64,
          ctx_min=1024, ctx_max=32768, gen=128, chunk=2048, seed=505)


def make_decoder_weights(shape: DecoderShape, seed: int, w_std: float = 0.02,
                         random_gains: bool = False) -> dict:
    """Random-init decoder weights, bf16 bits.

    Layout (row-major, PyTorch ``nn.Linear`` convention W[out, in]):
      embed [V, d]; per layer: attn_norm [d], wqkv [(Hq + 2 Hkv) hd, d] (q rows,
      then k rows, then v rows), wo [d, Hq hd], ffn_norm [d], w13 [2F, d]
      (gate rows then up rows), w2 [d, F]; final_norm [d]; lm_head [V, d].
    Norm gains are 1.0 unless ``random_gains`` (then 1 + N(0, 0.1^2)).
    """
    rng = np.random.default_rng(seed)
    s = shape
    nqkv = (s.n_heads_q + 2 * s.n_heads_kv) * s.head_dim
    one = to_bf16_bits(np.ones(s.d, np.float32))

    def gain():
        if not random_gains:
            return one.copy()
        return to_bf16_bits(1.0 + 0.1 * rng.standard_normal(s.d, dtype=np.float32))

    w = {"embed": normal_bf16(rng, (s.vocab, s.d), w_std), "layers": []}
    for _ in range(s.n_layers):
        w["layers"].append({
            "attn_norm": gain(),
            "wqkv": normal_bf16(rng, (nqkv, s.d), w_std),
            "wo": normal_bf16(rng, (s.d, s.n_heads_q * s.head_dim), w_std),
            "ffn_norm": gain(),
            "w13": normal_bf16(rng, (2 * s.ffn, s.d), w_std),
            "w2": normal_bf16(rng, (s.d, s.ffn), w_std),
        })
    w["final_norm"] = gain()
    w["lm_head"] = normal_bf16(rng, (s.vocab, s.d), w_std)
    return w


def make_prompts(n_seq: int, min_len: int, max_len: int, vocab: int, seed: int):
    """Prompt lengths uniform in [min_len, max_len] and token ids uniform in [0, vocab)."""
    rng = np.random.default_rng(seed + 1)
    lens = rng.integers(min_len, max_len + 1, size=n_seq)
    return [rng.integers(0, vocab, size=int(n), dtype=np.int64).astype(np.int32) for n in lens]


def make_c5_prompt_lengths(n_seq: int, lo: int, hi: int, seed: int) -> np.ndarray:
    """Context lengths log-uniform in [lo, hi]: round(exp(U[ln lo, ln hi]))."""
    rng = np.random.default_rng(seed + 2)
    u = rng.uniform(math.log(lo), math.log(hi), size=n_seq)
    return np.clip(np.rint(np.exp(u)), lo, hi).astype(np.int64)


def make_logprob_head(n_rows: int, d: int, vocab: int, w_std: float, seed: int,
                      h_std: float = 1.0, random_gain: bool = False) -> dict:
    """Hidden states h [n_rows, d] ~ N(0, h_std^2), lm_head [vocab, d] ~ N(0, w_std^2),
    norm gain [d] (ones unless random_gain) and target ids uniform in [0, vocab)."""
    rng = np.random.default_rng(seed)
    h = normal_bf16(rng, (n_rows, d), h_std)
    w = normal_bf16(rng, (vocab, d), w_std)
    if random_gain:
        g = to_bf16_bits(1.0 + 0.1 * rng.standard_normal(d, dtype=np.float32))
    else:
        g = to_bf16_bits(np.ones(d, np.float32))
    ids = rng.integers(0, vocab, size=n_rows).astype(np.int32)
    return {"h": h, "w": w, "gain": g, "ids": ids}


def make_moe_layer(n_tokens: int, d: int, ffn: int, n_experts: int, w_std: float,
                   seed: int, router_std: float = 1.0) -> dict:
    """x [T, d] ~ N(0,1) bf16; router logits [T, E] ~ N(0, router_std^2) fp32;
    w13 [E, 2F, d] (gate rows then up rows) and w2 [E, d, F] ~ N(0, w_std^2) bf16."""
    rng = np.random.default_rng(seed)
    x = normal_bf16(rng, (n_tokens, d), 1.0)
    logits = (router_std * rng.standard_normal((n_tokens, n_experts), dtype=np.float32)).astype(np.float32)
    w13 = normal_bf16(rng, (n_experts, 2 * ffn, d), w_std)
    w2 = normal_bf16(rng, (n_experts, d, ffn), w_std)
    return {"x": x, "router_logits": logits, "w13": w13, "w2": w2}
