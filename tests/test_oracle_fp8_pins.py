"""Pins of the block-FP8 oracle against things other than itself: torch's e4m3fn
conversion (a library routine), the format's closed forms, the half-ulp error bound,
exact round trips, block independence, and the GEMM against a block-wise promotion
restatement and an fp64 triple loop."""
import numpy as np
import pytest
import torch

from oracle import fp8


def test_code_table_closed_forms():
    v = fp8.e4m3_values()
    assert v[0x7E] == 448.0 and np.isnan(v[0x7F]) and np.isnan(v[0xFF])
    assert v[0x01] == 2.0 ** -9 and v[0x08] == 2.0 ** -6 and v[0x38] == 1.0
    assert v[0xC0] == -2.0 and v[0x80] == 0.0 and np.signbit(v[0x80])
    finite = v[~np.isnan(v)]
    assert len(finite) == 254 and len(np.unique(finite)) == 253    # +0 and -0 compare equal


def test_encode_matches_torch_e4m3fn_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000) * 30,
        rng.standard_normal(5000) * 1e-2,                       # subnormal range
        fp8.e4m3_values()[:0x7E].astype(np.float64),            # every positive code exactly
        (fp8.e4m3_values()[:0x7E] + fp8.e4m3_values()[1:0x7F]) / 2,   # every midpoint: ties
        [0.0, -0.0, 448.0, -448.0, 2.0 ** -10, 3 * 2.0 ** -10],
    ])
    x = x[np.abs(x) <= 448].astype(np.float32)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(fp8.e4m3_encode(x), want)


def test_encode_saturates_and_decodes():
    assert fp8.e4m3_encode(np.array([500.0, -1e9])).tolist() == [0x7E, 0xFE]
    x = np.array([1.0625, 1.1875, -3.0, 0.0], np.float32)     # ties to even mantissa
    assert fp8.e4m3_decode(fp8.e4m3_encode(x)).tolist() == [1.0, 1.25, -3.0, 0.0]


def test_scale_rule_and_error_bound():
    rng = np.random.default_rng(2)
    for amax in [1e-30, 1e-3, 0.7, 1.0, 448.0, 449.0, 3e4]:
        s = float(fp8.block_scale(np.float64(amax)))
        assert np.log2(s) == np.round(np.log2(s))              # a power of two
        assert 224.0 < amax / s <= 448.0
    assert float(fp8.block_scale(np.float64(0.0))) == 1.0
    x = (rng.standard_normal((4, 256)) * 5).astype(np.float32)
    q, s = fp8.quantize_act(x)
    dq = fp8.dequantize_blocks(q, s, 1)
    # 3 mantissa bits: error <= 2^-4 relative for normals, <= half the subnormal step otherwise
    sub = np.repeat(s, 128, axis=1) * 2.0 ** -10
    assert np.all(np.abs(dq - x) <= np.maximum(np.abs(x) * 2.0 ** -4, sub) + 1e-30)
    # values already on the grid survive the round trip exactly
    q2, s2 = fp8.quantize_act(dq)
    assert np.array_equal(fp8.dequantize_blocks(q2, s2, 1), dq)


def test_blocks_are_independent():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((256, 384)).astype(np.float32)
    q, s = fp8.quantize_weight(w)
    assert s.shape == (2, 3)
    w2 = w.copy()
    w2[:128, :128] *= 1000.0                                 # only block (0, 0) changes
    q2, s2 = fp8.quantize_weight(w2)
    assert s2[0, 0] != s[0, 0] and np.array_equal(np.delete(s2.ravel(), 0), np.delete(s.ravel(), 0))
    assert np.array_equal(q2[128:], q[128:]) and np.array_equal(q2[:128, 128:], q[:128, 128:])
    a = rng.standard_normal((3, 256)).astype(np.float32)
    qa, sa = fp8.quantize_act(a)
    qb, sb = fp8.quantize_act(a[1:2])                         # one row alone: same codes and scales
    assert np.array_equal(qb, qa[1:2]) and np.array_equal(sb, sa[1:2])


def test_gemm_equals_blockwise_promotion_and_triple_loop():
    rng = np.random.default_rng(4)
    M, N, K = 5, 256, 384
    a = (rng.standard_normal((M, K)) * 3).astype(np.float32)
    w = (rng.standard_normal((N, K)) * 0.05).astype(np.float32)
    qa, sa = fp8.quantize_act(a)
    qw, sw = fp8.quantize_weight(w)
    got = fp8.gemm_fp8(qa, sa, qw, sw)
    va, vw = fp8.e4m3_decode(qa).astype(np.float64), fp8.e4m3_decode(qw).astype(np.float64)
    prom = np.zeros((M, N))
    for kb in range(K // 128):                               # the kernel's grouping: per-block sums, then scales
        part = va[:, kb * 128:(kb + 1) * 128] @ vw[:, kb * 128:(kb + 1) * 128].T
        prom += part * sa[:, kb:kb + 1] * np.repeat(sw[:, kb], 128)[None, :N]
    assert np.allclose(got, prom, rtol=1e-6, atol=1e-6)
    m, n = 2, 131
    ref = sum(float(va[m, k]) * float(sa[m, k // 128]) * float(vw[n, k]) * float(sw[n // 128, k // 128])
              for k in range(K))
    assert abs(float(got[m, n]) - ref) <= 1e-6 * max(1.0, abs(ref))
    # and close to the unquantised product (block-FP8 error, a few percent of sum|a||w|)
    assert np.max(np.abs(got - a @ w.T) / (np.abs(a) @ np.abs(w).T)) < 0.1
