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


def bf16_close(got: np.ndarray, want: np.ndarray, ulps: float = 1.0, frac_exact: float = 0.95, atol: float = 0.0):
    """got within `ulps` bf16 ulps (relative 2^-8 per ulp) of want, and mostly bit-equal."""
    tol = ulps * 2.0 ** -7 * np.abs(want) + atol
    bad = np.abs(got - want) > tol
    assert not bad.any(), f"{bad.sum()} elements beyond {ulps} bf16 ulp; max err {np.max(np.abs(got - want))}"
    assert np.mean(got == want) >= frac_exact, f"only {np.mean(got == want):.3f} bit-equal"
