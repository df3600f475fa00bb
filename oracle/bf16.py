"""bf16 rounding used by the oracle (test infrastructure only).

bf16 keeps the top 16 bits of an IEEE fp32 value.  Rounding is to nearest,
ties to even, which is the rounding the article's numerical contract leaves
implicit ([Article] §2, "same quantization and rounding"; one rounding per
boundary in §4.4, condition 3).  NaN stays NaN; overflow rounds to +-inf.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own.
"""
import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round fp32 values to the nearest bf16 value (ties to even); returns fp32."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) & np.uint64(0xFFFF0000)
    out = r.astype(np.uint32).view(np.float32).copy()
    nan = np.isnan(x)
    if nan.any():
        out[nan] = np.float32(np.nan)
    return out.reshape(x.shape)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """bf16 bit patterns (uint16) -> exact fp32 values."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).reshape(b.shape)


def f32_to_bf16_bits(x) -> np.ndarray:
    """fp32 values (already bf16-exact or not) -> bf16 bit patterns after RNE rounding."""
    r = round_bf16(x)
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
