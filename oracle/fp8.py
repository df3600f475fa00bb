"""Block-FP8 (e4m3) quantisation and the W8A8 GEMM it feeds (test infrastructure only).

[Article] §4.1 ("Dense GEMM: keep FP8, one accumulation order for every M"):
the deployed model is block FP8, the inference GEMM is W8A8, and every training
forward quantises the bf16 master weights to block FP8 by the deployment rule
before calling the same GEMM.

Readings where the pages are silent (the plainest ones the rest supports):
  * Element format: e4m3 "fn" (1 sign, 4 exponent bits with bias 7, 3 mantissa
    bits, no infinities, largest finite 448).  Conversion rounds to nearest,
    ties to the even code, keeps the sign (also of zero) and saturates at +-448.
  * Blocks: 128 x 128 for weights [N, K]; 1 x 128 (one row, 128 consecutive K)
    for activations [M, K].  K is a multiple of 128.
  * Scale of a block: the power of two s = 2^ceil(log2(amax / 448)) (s = 1 for
    an all-zero block), so that every |x| / s <= 448 and dequantisation
    q * s is exact in fp32 and bf16.  Power-of-two (UE8M0) scales are the form
    the Blackwell deployment GEMMs take.
  * GEMM: C[m, n] = sum_k (qa[m, k] sa[m, k/128]) (qw[n, k] sw[n/128, k/128]),
    the product of the dequantised operands (the block-wise promotion a kernel
    does is the same sum regrouped, exact for power-of-two scales); fp32
    output, or bf16 rounded once.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own.
"""
from __future__ import annotations

import numpy as np

from .bf16 import round_bf16

E4M3_MAX = 448.0


def e4m3_values() -> np.ndarray:
    """Value of every 8-bit e4m3fn code, NaN for the two NaN codes (0x7F, 0xFF)."""
    v = np.empty(256, dtype=np.float64)
    for code in range(256):
        sign = -1.0 if code & 0x80 else 1.0
        e = (code >> 3) & 0xF
        m = code & 0x7
        if e == 0xF and m == 0x7:
            v[code] = np.nan
        elif e == 0:
            v[code] = sign * (m / 8.0) * 2.0 ** -6
        else:
            v[code] = sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)
    return v


_VALUES = e4m3_values()
_POS_CODES = np.arange(0, 0x7F)            # 0x00 .. 0x7E: +0 .. 448, increasing
_POS_VALUES = _VALUES[_POS_CODES]


def e4m3_encode(x) -> np.ndarray:
    """fp32/fp64 values -> e4m3 codes (uint8): nearest value, ties to the even code, saturating at 448."""
    x = np.asarray(x, dtype=np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.searchsorted(_POS_VALUES, a, side="left")          # first value >= a
    hi = np.minimum(hi, len(_POS_VALUES) - 1)
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - _POS_VALUES[lo], _POS_VALUES[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (_POS_CODES[hi] % 2 == 0) & (hi != lo))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.int64)
    code = np.where(a == _POS_VALUES[hi], _POS_CODES[hi], code)
    return (code | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)   # the sign is kept, also on zero


def e4m3_decode(codes) -> np.ndarray:
    return _VALUES[np.asarray(codes, dtype=np.int64)].astype(np.float32)


def block_scale(amax) -> np.ndarray:
    """Power-of-two scale of a block with absolute maximum amax (1 for an all-zero block)."""
    amax = np.asarray(amax, dtype=np.float64)
    out = np.ones_like(amax)
    nz = amax > 0
    out[nz] = 2.0 ** np.ceil(np.log2(amax[nz] / E4M3_MAX))
    return out.astype(np.float32)


def quantize_blocks(x, block_rows: int, block_cols: int = 128):
    """x [R, C] (C a multiple of block_cols) -> (codes uint8 [R, C], scales fp32 [ceil(R/br), C/bc])."""
    x = np.asarray(x, dtype=np.float32)
    R, C = x.shape
    assert C % block_cols == 0
    nbr = -(-R // block_rows)
    scales = np.empty((nbr, C // block_cols), dtype=np.float32)
    codes = np.empty((R, C), dtype=np.uint8)
    for i in range(nbr):
        r0, r1 = i * block_rows, min(R, (i + 1) * block_rows)
        for j in range(C // block_cols):
            blk = x[r0:r1, j * block_cols:(j + 1) * block_cols]
            s = block_scale(np.max(np.abs(blk)))
            scales[i, j] = s
            codes[r0:r1, j * block_cols:(j + 1) * block_cols] = e4m3_encode(blk.astype(np.float64) / float(s))
    return codes, scales


def dequantize_blocks(codes, scales, block_rows: int, block_cols: int = 128) -> np.ndarray:
    v = e4m3_decode(codes).astype(np.float64)
    R, C = v.shape
    s = np.repeat(np.repeat(scales.astype(np.float64), block_rows, axis=0)[:R], block_cols, axis=1)[:, :C]
    return (v * s).astype(np.float32)


def quantize_act(x):
    """Activations [M, K]: 1 x 128 blocks."""
    return quantize_blocks(x, 1)


def quantize_weight(w):
    """Weights [N, K]: 128 x 128 blocks."""
    return quantize_blocks(w, 128)


def gemm_fp8(qa, sa, qw, sw, out: str = "fp32") -> np.ndarray:
    """W8A8 GEMM: the fp64 product of the dequantised operands, then fp32 (or bf16)."""
    a = dequantize_blocks(qa, sa, 1).astype(np.float64)
    w = dequantize_blocks(qw, sw, 128).astype(np.float64)
    c = (a @ w.T).astype(np.float32)
    return round_bf16(c) if out == "bf16" else c
