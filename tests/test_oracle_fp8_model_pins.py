"""Pins of the block-FP8 decoder oracle (W8A8 linear layers and the FP8 K/V round
trip of "vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 and §4.2) against
what the mathematics of power-of-two block scaling fixes: the reduction of the
W8A8 layer to a plain fp64 matmul when both operands already sit on the FP8 grid,
scale equivariance row by row and K block by K block, the round trip's grid,
error bound and per-(token, head) independence, and the residual wiring of the
layer."""
import numpy as np

from oracle import fp8, model, ops
from oracle.bf16 import round_bf16
from synthetic import DecoderShape, make_decoder_weights

E4M3 = fp8.e4m3_values()


def _on_grid(rng, rows, cols, block_rows, exps):
    """Values of e4m3 codes times a power of two per (block_rows x 128) block, each
    block's largest magnitude exactly 448 times its scale (so the block's scale
    is that power of two and quantisation is the identity)."""
    codes = rng.integers(0, 0x7F, (rows, cols))
    codes[codes == 0x7F] = 0x7E
    sign = np.where(rng.random((rows, cols)) < 0.5, -1.0, 1.0)
    x = E4M3[codes] * sign
    for i in range(0, rows, block_rows):
        for j in range(0, cols, 128):
            e = exps[(i // block_rows) % len(exps), (j // 128) % exps.shape[1]]
            x[i:i + block_rows, j:j + 128] *= 2.0 ** e
            x[i, j] = 448.0 * 2.0 ** e
    return x.astype(np.float32)


def test_linear_fp8_on_grid_operands_is_the_plain_matmul():
    rng = np.random.default_rng(1)
    exps_a = rng.integers(-12, -4, (5, 3))
    exps_w = rng.integers(-14, -6, (3, 3))
    a = _on_grid(rng, 5, 384, 1, exps_a)
    w = _on_grid(rng, 256, 384, 128, exps_w)
    assert np.array_equal(round_bf16(a), a) and np.array_equal(round_bf16(w), w)   # bf16 inputs too
    qw, sw = fp8.quantize_weight(w)
    assert np.array_equal(np.log2(sw), exps_w[:2, :3].astype(np.float32))
    got = model.linear_fp8(a, qw, sw)
    want = round_bf16((a.astype(np.float64) @ w.astype(np.float64).T).astype(np.float32))
    assert np.array_equal(got, want)


def test_linear_fp8_scale_equivariance():
    """A power of two on a row of x scales that output row by the same power
    (rows are quantised alone); 2^j on one 128-column block of x with 2^-j on the
    same columns of W changes nothing (the K blocks are quantised alone)."""
    rng = np.random.default_rng(2)
    x = round_bf16(rng.standard_normal((6, 384)).astype(np.float32))
    w = round_bf16((rng.standard_normal((256, 384)) * 0.05).astype(np.float32))
    qw, sw = fp8.quantize_weight(w)
    y = model.linear_fp8(x, qw, sw)
    f = 2.0 ** np.array([0, 3, -5, 7, -2, 1], np.float32)[:, None]
    assert np.array_equal(model.linear_fp8(x * f, qw, sw), y * f)
    x2, w2 = x.copy(), w.copy()
    x2[:, 128:256] *= 2.0 ** 6
    w2[:, 128:256] *= 2.0 ** -6
    assert np.array_equal(model.linear_fp8(x2, *fp8.quantize_weight(w2)), y)
    # the W8A8 layer is not the bf16 layer: quantisation really happens, and with the
    # identity as weight (on the FP8 grid) the output is the activation's own round trip
    assert not np.array_equal(y, ops.linear(x, w))
    eye = np.eye(384, dtype=np.float32)
    qa, sa = fp8.quantize_act(x)
    assert np.array_equal(model.linear_fp8(x, *fp8.quantize_weight(eye)), fp8.dequantize_blocks(qa, sa, 1))


def test_kv_round_trip_grid_bound_and_independence():
    rng = np.random.default_rng(3)
    t = round_bf16((rng.standard_normal((40, 3, 64)) * np.exp(rng.standard_normal((40, 3, 1)) * 3)).astype(np.float32))
    t[5, 1] = 0.0
    out = model.kv_round_trip(t)
    amax = np.abs(t).max(-1)
    for i in range(40):
        for h in range(3):
            if amax[i, h] == 0:
                assert np.all(out[i, h] == 0)
                continue
            s = 2.0 ** np.ceil(np.log2(amax[i, h] / 448.0))
            codes = out[i, h] / s
            assert np.all(np.isin(np.abs(codes), E4M3[:0x7F]))          # on the e4m3 grid of its own scale
            assert 224.0 <= np.abs(codes).max() <= 448.0                    # amax / s in (224, 448], then rounded
            err = np.abs(out[i, h] - t[i, h])
            assert np.all(err <= np.maximum(np.abs(t[i, h]) * 2.0 ** -4, s * 2.0 ** -10))
    # one vector's values move no other vector's result
    t2 = t.copy()
    t2[7, 2] *= 1000.0
    out2 = model.kv_round_trip(t2)
    keep = np.ones((40, 3), bool)
    keep[7, 2] = False
    assert np.array_equal(out2[keep], out[keep])
    assert np.array_equal(model.kv_round_trip(out), out)                # idempotent


def test_fp8_layer_residual_wiring_and_distance_from_bf16():
    shape = DecoderShape(2, 256, 4, 2, 64, 256, 512)
    W = model.weights_to_f32(make_decoder_weights(shape, seed=5, w_std=0.05))
    W8 = model.fp8_weights(W)
    rng = np.random.default_rng(6)
    r = round_bf16(rng.standard_normal((20, 256)).astype(np.float32))
    pos = np.arange(20)
    # with the attention and FFN output projections zero the layer is the identity on r
    lz = dict(W["layers"][0])
    lz["wo"] = np.zeros_like(lz["wo"])
    lz["w2"] = np.zeros_like(lz["w2"])
    lz8 = model.fp8_weights({"layers": [lz]})["layers"][0]
    assert np.array_equal(model.layer(lz8, shape, r, pos), r)
    # the FP8 layer is near the bf16 layer but not equal to it: every W8A8 GEMM input
    # carries at most 2^-4 relative error, so the two sub-layer outputs differ by a
    # few percent of their size
    out8, o8, dn8 = model.layer(W8["layers"][0], shape, r, pos, return_parts=True)
    out, o, dn = model.layer(W["layers"][0], shape, r, pos, return_parts=True)
    assert not np.array_equal(o8, o) and not np.array_equal(dn8, dn)
    for a, b in ((o8, o), (dn8, dn)):
        rel = np.linalg.norm(a - b) / np.linalg.norm(b)
        assert 1e-3 < rel < 0.1, rel


def test_fp8_layer_first_token_reads_its_own_round_tripped_v():
    """At position 0 attention has one key, so its output is the token's own V as
    read back from the FP8 cache; with Wo the identity (on the FP8 grid) the
    attention sub-layer output is that V requantised in 1 x 128 blocks.  hd 64
    puts two kv heads with different scales in one 128-column block."""
    shape = DecoderShape(1, 256, 4, 4, 64, 256, 512)
    W = model.weights_to_f32(make_decoder_weights(shape, seed=7, w_std=0.05))
    lw = dict(W["layers"][0])
    lw["wo"] = np.eye(256, dtype=np.float32)
    lw["wqkv"][512:512 + 64] *= 16.0                     # kv head 0 of V much larger than head 1
    l8 = model.fp8_weights({"layers": [lw]})["layers"][0]
    r = round_bf16(np.random.default_rng(8).standard_normal((1, 256)).astype(np.float32))
    _, o, _ = model.layer(l8, shape, r, np.arange(1), return_parts=True)
    x, _ = ops.rmsnorm(r, lw["attn_norm"], shape.eps)
    v = model.linear_fp8(x, *l8["fp8"]["wqkv"])[:, 512:].reshape(1, 4, 64)
    v_read = model.kv_round_trip(v).reshape(1, 256)
    q, s = fp8.quantize_act(v_read)
    assert np.array_equal(o, fp8.dequantize_blocks(q, s, 1))
    assert not np.array_equal(model.kv_round_trip(v), v)          # the round trip is not the identity here


def test_fp8_layer_attention_mixes_round_tripped_k_and_v():
    """With several keys the attention output mixes V vectors, so the FP8 round
    trips of K (after RoPE) and V are visible through the O projection's own
    1 x 128 quantisation: with Wo the identity, the attention sub-layer output is
    the activation round trip of attention(q, rt(rope(k)), rt(v)), and neither the
    bf16 V, the bf16 K nor K quantised before its rotation gives it."""
    shape = DecoderShape(1, 256, 4, 2, 64, 256, 512)
    W = model.weights_to_f32(make_decoder_weights(shape, seed=9, w_std=0.05))
    lw = dict(W["layers"][0])
    lw["wo"] = np.eye(256, dtype=np.float32)
    l8 = model.fp8_weights({"layers": [lw]})["layers"][0]
    L = 5
    pos = np.arange(L)
    r = round_bf16(np.random.default_rng(10).standard_normal((L, 256)).astype(np.float32))
    _, o, _ = model.layer(l8, shape, r, pos, return_parts=True)
    x, _ = ops.rmsnorm(r, lw["attn_norm"], shape.eps)
    qkv = model.linear_fp8(x, *l8["fp8"]["wqkv"])
    q = ops.rope(qkv[:, :256].reshape(L, 4, 64), pos, shape.rope_theta)
    k_raw = qkv[:, 256:384].reshape(L, 2, 64)
    k = ops.rope(k_raw, pos, shape.rope_theta)
    v = qkv[:, 384:].reshape(L, 2, 64)

    def o_of(kk, vv):
        a = ops.attention(q, kk, vv, pos).reshape(L, 256)
        qa, sa = fp8.quantize_act(a)
        return fp8.dequantize_blocks(qa, sa, 1)

    rt = model.kv_round_trip
    assert np.array_equal(o, o_of(rt(k), rt(v)))
    assert not np.array_equal(o, o_of(rt(k), v))
    assert not np.array_equal(o, o_of(k, rt(v)))
    assert not np.array_equal(o, o_of(ops.rope(rt(k_raw), pos, shape.rope_theta), rt(v)))
