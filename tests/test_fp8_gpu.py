"""Block-FP8 quantisation and the W8A8 tcgen05 GEMM ([Article] §4.1) through the C ABI:
codes and scales bit-exact against the oracle, the GEMM within fp32 accumulation of
the oracle's exact product, and every row's result independent of the batch.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own."""
import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from oracle import fp8 as ofp8
from synthetic import bits_to_f32, normal_bf16
from tests.gpu_util import dev_bf16, same_bits

pytestmark = pytest.mark.gpu


def _quant(xb, block_rows):
    R, C = xb.shape
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    s = torch.empty((-(-R // block_rows), C // 128), dtype=torch.float32, device="cuda")
    bi.bi_quantize_fp8(dev_bf16(xb), R, C, block_rows, q, s)
    return q, s


@pytest.mark.parametrize("R,C,br", [(1, 128, 1), (37, 384, 1), (256, 512, 128), (300, 256, 128), (5, 1024, 128)])
def test_quantize_matches_oracle_bitwise(R, C, br):
    rng = np.random.default_rng(R * C + br)
    xb = normal_bf16(rng, (R, C), 3.0)
    xf = bits_to_f32(xb).copy()
    xf[0, :7] = [0.0, -0.0, 1e-38, -3e-39, 6e4, -6e4, 2.0 ** -133]    # zeros, subnormals, large values
    xf[min(R - 1, 2), 128:256 if C >= 256 else 128] = 0.0              # an all-zero block where there is one
    from synthetic import to_bf16_bits
    xb = to_bf16_bits(xf)
    q, s = _quant(xb, br)
    want_q, want_s = ofp8.quantize_blocks(bits_to_f32(xb), br)
    assert np.array_equal(s.cpu().numpy(), want_s)
    assert np.array_equal(q.cpu().numpy(), want_q)


def _fp8_operands(rng, M, N, K, a_std=1.0, w_std=0.05):
    ab, wb = normal_bf16(rng, (M, K), a_std), normal_bf16(rng, (N, K), w_std)
    qa, sa = _quant(ab, 1)
    qw, sw = _quant(wb, 128)
    return qa, sa, qw, sw


@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (5, 256, 512), (130, 384, 256), (300, 1024, 1024), (64, 3072, 2048)])
def test_gemm_fp8_parity(M, N, K):
    rng = np.random.default_rng(M + N + K)
    qa, sa, qw, sw = _fp8_operands(rng, M, N, K)
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    bi.bi_gemm_fp8(qa, sa, M, K, qw, sw, N, C32, bi.BI_DTYPE_FP32)
    want = ofp8.gemm_fp8(qa.cpu().numpy(), sa.cpu().numpy(), qw.cpu().numpy(), sw.cpu().numpy())
    a = ofp8.dequantize_blocks(qa.cpu().numpy(), sa.cpu().numpy(), 1).astype(np.float64)
    w = ofp8.dequantize_blocks(qw.cpu().numpy(), sw.cpu().numpy(), 128).astype(np.float64)
    absdot = np.abs(a) @ np.abs(w).T
    # fp32 accumulation in another order: within a small multiple of 2^-24 sum|a||w|
    assert np.max(np.abs(C32.cpu().numpy() - want) / (absdot + 1e-30)) < 1e-5
    Cb = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm_fp8(qa, sa, M, K, qw, sw, N, Cb, bi.BI_DTYPE_BF16)
    # the bf16 output is the fp32 result rounded once
    assert same_bits(Cb, C32.to(torch.bfloat16))
    assert bi.bi_device_status() == 0


@pytest.mark.parametrize("N,K", [(256, 512), (512, 1408), (3072, 2048), (20480, 256)])
def test_gemm_fp8_rows_invariant_to_M_and_order(N, K):
    rng = np.random.default_rng(N)
    qa, sa, qw, sw = _fp8_operands(rng, 300, N, K)
    full = torch.empty((300, N), dtype=torch.float32, device="cuda")
    bi.bi_gemm_fp8(qa, sa, 300, K, qw, sw, N, full, bi.BI_DTYPE_FP32)
    for M in (1, 7, 16, 17, 33, 64, 65, 127, 128, 129, 255):
        off = 300 - M
        part = torch.empty((M, N), dtype=torch.float32, device="cuda")
        bi.bi_gemm_fp8(qa[off:].contiguous(), sa[off:].contiguous(), M, K, qw, sw, N, part, bi.BI_DTYPE_FP32)
        assert same_bits(part, full[off:]), M
    perm = torch.from_numpy(rng.permutation(300)).cuda()
    outp = torch.empty_like(full)
    bi.bi_gemm_fp8(qa[perm].contiguous(), sa[perm].contiguous(), 300, K, qw, sw, N, outp, bi.BI_DTYPE_FP32)
    assert same_bits(outp, full[perm])


def test_training_side_requantisation_is_deterministic():
    """The training forward requantises the bf16 master weights every call: the
    codes and scales are bitwise the same each time and match the oracle."""
    rng = np.random.default_rng(7)
    wb = normal_bf16(rng, (384, 640), 0.02)
    q1, s1 = _quant(wb, 128)
    q2, s2 = _quant(wb, 128)
    assert torch.equal(q1, q2) and torch.equal(s1, s2)


@pytest.mark.parametrize("rows,d,resid", [(1, 128, False), (37, 512, True), (64, 2048, True), (5, 16384, False),
                                          (130, 1408, True)])
def test_rmsnorm_fp8_equals_norm_then_quantize(rows, d, resid):
    """The fused norm + quantisation writes exactly what bi_rmsnorm followed by
    bi_quantize_fp8 writes: codes, scales, the bf16 row and the residual."""
    rng = np.random.default_rng(rows + d)
    x = dev_bf16(normal_bf16(rng, (rows, d), 2.0))
    g = dev_bf16(normal_bf16(rng, (d,), 1.0))
    r0 = dev_bf16(normal_bf16(rng, (rows, d), 1.0))
    r1, r2 = r0.clone(), r0.clone()
    y1 = torch.empty((rows, d), dtype=torch.bfloat16, device="cuda")
    bi.bi_rmsnorm(x, r1 if resid else None, g, y1, rows, d, 1e-6)
    q1 = torch.empty((rows, d), dtype=torch.uint8, device="cuda")
    s1 = torch.empty((rows, d // 128), dtype=torch.float32, device="cuda")
    bi.bi_quantize_fp8(y1, rows, d, 1, q1, s1)
    y2 = torch.empty_like(y1)
    q2, s2 = torch.empty_like(q1), torch.empty_like(s1)
    bi.bi_rmsnorm_fp8(x, r2 if resid else None, g, y2, q2, s2, rows, d)
    assert torch.equal(q1, q2) and same_bits(s1, s2) and same_bits(y1, y2) and same_bits(r1, r2)
    q3, s3 = torch.empty_like(q1), torch.empty_like(s1)
    r3 = r0.clone()
    bi.bi_rmsnorm_fp8(x, r3 if resid else None, g, None, q3, s3, rows, d)      # no bf16 row written
    assert torch.equal(q1, q3) and same_bits(s1, s3) and same_bits(r1, r3)


@pytest.mark.parametrize("T,F", [(1, 128), (33, 1536), (300, 512), (7, 5632)])
def test_swiglu_fp8_matches_oracle(T, F):
    """SiLU-mul-quant: codes and scales of bf16(silu(g) u) by the oracle's rule; a
    code may differ only where the kernel's exp and numpy's exp round the product
    to different bf16 values (one e4m3 step at most, and rarely)."""
    from oracle import ops
    rng = np.random.default_rng(T * F)
    g13 = normal_bf16(rng, (T, 2 * F), 2.0)
    q = torch.empty((T, F), dtype=torch.uint8, device="cuda")
    s = torch.empty((T, F // 128), dtype=torch.float32, device="cuda")
    bi.bi_swiglu_fp8(dev_bf16(g13), T, F, q, s)
    gf = bits_to_f32(g13)
    a = ops.silu_mul(gf[:, :F], gf[:, F:])
    wq, ws = ofp8.quantize_act(a)
    gq, gs = q.cpu().numpy(), s.cpu().numpy()
    assert np.mean(gs == ws) >= 0.999
    same_scale = np.repeat(gs == ws, 128, axis=1)
    diff = (gq != wq) & same_scale
    assert np.mean(gq == wq) >= 0.999
    assert np.all(np.abs(gq[diff].astype(np.int32) - wq[diff].astype(np.int32)) <= 1)
