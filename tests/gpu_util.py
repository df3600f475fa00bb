"""Helpers shared by the GPU tests (device transfer of bf16 bit arrays, bit-exact compares)."""
import numpy as np
import torch

from synthetic import bits_to_f32, to_bf16_bits

DEV = "cuda"


def dev_bf16(bits) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(DEV)


def dev_bf16_from_f32(x) -> torch.Tensor:
    return dev_bf16(to_bf16_bits(np.asarray(x, np.float32)))


def host_f32(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return bits_to_f32(t.view(torch.int16).cpu().numpy().view(np.uint16))
    return t.float().cpu().numpy()


def same_bits(a: torch.Tensor, b: torch.Tensor) -> bool:
    if a.shape != b.shape or a.dtype != b.dtype:
        return False
    if a.dtype in (torch.bfloat16, torch.float16):
        return torch.equal(a.view(torch.int16), b.view(torch.int16))
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


def bf16_ulp(x) -> np.ndarray:
    """One bf16 ulp at each |x|: 2^(e - 7) for |x| in [2^e, 2^(e+1)) (8 significant
    bits), and 2^-133 (the smallest subnormal step) below 2^-126 and at zero."""
    a = np.abs(np.asarray(x, np.float64))
    _, e = np.frexp(a)                       # a = f * 2^e with f in [0.5, 1)
    e = np.where(a == 0, -125, np.maximum(e, -125))
    return np.ldexp(1.0, e - 8)


def bf16_close(got: np.ndarray, want: np.ndarray, ulps: float = 1.0, frac_exact: float = 0.95, atol: float = 0.0):
    """got within `ulps` bf16 ulps of want (one ulp measured exactly at |want|), plus
    atol, and at least `frac_exact` of the elements bit-equal."""
    tol = ulps * bf16_ulp(want) + atol
    bad = np.abs(np.asarray(got, np.float64) - np.asarray(want, np.float64)) > tol
    assert not bad.any(), f"{bad.sum()} elements beyond {ulps} bf16 ulp; max err {np.max(np.abs(got - want))}"
    assert np.mean(got == want) >= frac_exact, f"only {np.mean(got == want):.3f} bit-equal"
