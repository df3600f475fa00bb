"""Pins for the CPU oracle: closed forms, invariants, library routines and brute force.

Nothing here compares the oracle with itself.  Each test fixes a value the
mathematics (or an independent library routine) determines, chosen so that a
plausible slip in the oracle (a dropped term, a transposed operand, a wrong
sign, index or constant) fails at least one of them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as TF

import oracle
from oracle import ops, moe, model
from oracle.bf16 import round_bf16, bf16_bits_to_f32, f32_to_bf16_bits
from synthetic import DecoderShape, make_decoder_weights, to_bf16_bits, bits_to_f32

F32 = np.float32


def bf16_vals(rng, shape, std=1.0):
    return bits_to_f32(to_bf16_bits(rng.standard_normal(shape).astype(F32) * F32(std)))


def torch_bf16(x64: torch.Tensor) -> torch.Tensor:
    """Round through torch's bf16 conversion (fp64 -> fp32 -> bf16 -> fp64)."""
    return x64.to(torch.float32).to(torch.bfloat16).to(torch.float64)


# ----------------------------------------------------------------------------- bf16
def test_round_bf16_matches_torch_conversion():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(100000).astype(F32) * F32(1000),
        rng.standard_normal(1000).astype(F32) * F32(1e-40),        # subnormals
        np.array([0.0, -0.0, np.inf, -np.inf, 3.0e38, -3.0e38, 1.0, 1.00390625, 1.01171875], F32),
    ])
    # exact ties: bf16 value + half an ulp
    ties = (bits_to_f32(rng.integers(0x3000, 0x5000, 2000).astype(np.uint16)).view(np.uint32) | np.uint32(0x8000)).view(F32)
    x = np.concatenate([x, ties])
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    got = round_bf16(x)
    assert np.array_equal(got.view(np.uint32), want.view(np.uint32))
    assert np.isnan(round_bf16(np.array([np.nan], F32))[0])
    assert np.array_equal(bf16_bits_to_f32(f32_to_bf16_bits(x)).view(np.uint32), want.view(np.uint32))


# ----------------------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("c", [0.75, -3.0, 1e-3])
def test_rmsnorm_constant_row_closed_form(c):
    rng = np.random.default_rng(1)
    d = 256
    g = bf16_vals(rng, d) + F32(1.0)
    g = round_bf16(g)
    x = np.full((3, d), c, F32)
    x = round_bf16(x)
    cb = float(x[0, 0])
    y, r = ops.rmsnorm(x, g, 1e-6)
    want = cb / math.sqrt(cb * cb + 1e-6) * g.astype(np.float64)
    assert np.allclose(y[0], want, rtol=2 ** -7, atol=0)
    assert np.array_equal(r, x)


def test_rmsnorm_matches_torch_rms_norm_fp64():
    rng = np.random.default_rng(2)
    x = bf16_vals(rng, (17, 320), 2.0)
    g = round_bf16(bf16_vals(rng, 320, 0.3) + F32(1.0))
    y, _ = ops.rmsnorm(x, g, 1e-6)
    ref = torch_bf16(TF.rms_norm(torch.from_numpy(x).double(), (320,), torch.from_numpy(g).double(), eps=1e-6)).numpy()
    # at most one bf16 rounding flip (fp32 vs fp64 before the rounding)
    assert np.all(np.abs(y - ref) <= 2 ** -7 * np.abs(ref) + 1e-30)
    assert np.mean(y == ref) > 0.98


def test_rmsnorm_power_of_two_scale_is_exact():
    rng = np.random.default_rng(3)
    x = bf16_vals(rng, (5, 128))
    g = round_bf16(bf16_vals(rng, 128, 0.5) + F32(1.0))
    y1, _ = ops.rmsnorm(x, g, 1e-6)
    y2, _ = ops.rmsnorm(x * F32(4.0), g, 16e-6)
    assert np.array_equal(y1, y2)


def test_rmsnorm_residual_add_is_one_bf16_rounding():
    rng = np.random.default_rng(4)
    a = bf16_vals(rng, (9, 64))
    b = bf16_vals(rng, (9, 64))
    g = np.ones(64, F32)
    _, r = ops.rmsnorm(b, g, 1e-6, residual=a)
    want = (torch.from_numpy(a).to(torch.bfloat16) + torch.from_numpy(b).to(torch.bfloat16)).float().numpy()
    assert np.array_equal(r, want)


# ----------------------------------------------------------------------------- GEMM
def test_linear_bruteforce_fp64_tiny():
    rng = np.random.default_rng(5)
    M, N, K = 3, 5, 7
    a = bf16_vals(rng, (M, K))
    w = bf16_vals(rng, (N, K))
    c = np.zeros((M, N))
    for m in range(M):
        for n in range(N):
            for k in range(K):
                c[m, n] += float(a[m, k]) * float(w[n, k])
    assert np.allclose(ops.linear(a, w, "fp32"), c, rtol=1e-6, atol=1e-6)
    got = ops.linear(a, w, "bf16")
    assert np.all(np.abs(got - c) <= 2 ** -8 * np.abs(c) + 1e-6)


def test_linear_identity_weight():
    rng = np.random.default_rng(6)
    a = bf16_vals(rng, (4, 16))
    assert np.array_equal(ops.linear(a, np.eye(16, dtype=F32)), a)


# ----------------------------------------------------------------------------- RoPE
def test_rope_position_zero_identity_and_pair_norms():
    rng = np.random.default_rng(7)
    x = bf16_vals(rng, (6, 3, 64))
    assert np.array_equal(ops.rope(x, np.zeros(6, np.int64)), x)
    pos = np.array([1, 7, 100, 513, 4095, 32767])
    y = ops.rope(x, pos)
    n0 = x[..., :32] ** 2 + x[..., 32:] ** 2
    n1 = y[..., :32] ** 2 + y[..., 32:] ** 2
    assert np.allclose(n0, n1, rtol=2e-2, atol=1e-4)


def test_rope_matches_complex_rotation():
    """(x1 + i x2) * exp(i * pos * base^(-2i/hd)) is the textbook form of rotate-half RoPE."""
    rng = np.random.default_rng(8)
    hd = 32
    x = bf16_vals(rng, (5, 2, hd))
    pos = np.array([0, 3, 17, 250, 3000])
    freq = 10000.0 ** (-np.arange(hd // 2) * 2.0 / hd)
    z = (x[..., : hd // 2] + 1j * x[..., hd // 2:]) * np.exp(1j * pos[:, None, None] * freq[None, None, :])
    want = np.concatenate([z.real, z.imag], axis=-1)
    got = ops.rope(x, pos)
    assert np.all(np.abs(got - want) <= 2 ** -8 * np.abs(want) + 1e-5)


def test_rope_unit_vector_closed_forms():
    hd = 64
    e0 = np.zeros((1, 1, hd), F32)
    e0[0, 0, 0] = 1.0
    y = ops.rope(e0, np.array([3]))
    assert abs(y[0, 0, 0] - math.cos(3.0)) < 4e-3 and abs(y[0, 0, 32] - math.sin(3.0)) < 4e-3
    eq = np.zeros((1, 1, hd), F32)
    eq[0, 0, 16] = 1.0                       # i = hd/4 -> theta = base^(-1/2) = 0.01
    y = ops.rope(eq, np.array([100]))
    assert abs(y[0, 0, 16] - math.cos(1.0)) < 4e-3 and abs(y[0, 0, 48] - math.sin(1.0)) < 4e-3


def test_rope_relative_position_property():
    rng = np.random.default_rng(9)
    q = bf16_vals(rng, (1, 1, 64))
    k = bf16_vals(rng, (1, 1, 64))
    d1 = float(np.sum(ops.rope(q, [12]) * ops.rope(k, [5])))
    d2 = float(np.sum(ops.rope(q, [1012]) * ops.rope(k, [1005])))
    assert abs(d1 - d2) < 3e-2 * max(1.0, abs(d1))


# ----------------------------------------------------------------------------- attention
def _sdpa_fp64(q, k, v, q_pos):
    """torch SDPA in fp64 with an explicit causal mask and GQA by repeating kv heads."""
    hq, hkv = q.shape[1], k.shape[1]
    qt = torch.from_numpy(q).double().permute(1, 0, 2)
    kt = torch.from_numpy(k).double().permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    vt = torch.from_numpy(v).double().permute(1, 0, 2).repeat_interleave(hq // hkv, dim=0)
    mask = torch.arange(k.shape[0])[None, :] <= torch.from_numpy(np.asarray(q_pos))[:, None]
    o = TF.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask)
    return o.permute(1, 0, 2).numpy()


def test_attention_matches_torch_sdpa_gqa():
    rng = np.random.default_rng(10)
    L, hq, hkv, hd = 40, 4, 2, 16
    q = bf16_vals(rng, (L, hq, hd))
    k = bf16_vals(rng, (L, hkv, hd))
    v = bf16_vals(rng, (L, hkv, hd))
    pos = np.arange(L)
    got = ops.attention(q, k, v, pos)
    want = _sdpa_fp64(q, k, v, pos)
    assert np.all(np.abs(got - want) <= 2 ** -8 * np.abs(want) + 2e-6)
    # a query block starting mid-sequence (decode-like rows) gives the same rows
    got_tail = ops.attention(q[30:], k, v, pos[30:])
    assert np.array_equal(got_tail, got[30:])


def test_attention_closed_forms():
    rng = np.random.default_rng(11)
    hd = 8
    k = bf16_vals(rng, (10, 1, hd))
    v = bf16_vals(rng, (10, 1, hd))
    q = bf16_vals(rng, (10, 1, hd))
    o = ops.attention(q, k, v, np.arange(10))
    assert np.array_equal(o[0], v[0])                       # single key -> o = v
    qz = np.zeros_like(q)
    oz = ops.attention(qz, k, v, np.arange(10))              # q = 0 -> uniform average
    for i in range(10):
        assert np.allclose(oz[i, 0], v[: i + 1, 0].astype(np.float64).mean(0), rtol=2 ** -8, atol=1e-6)
    ke = np.repeat(k[:1], 10, axis=0)                         # equal keys -> uniform average
    oe = ops.attention(q, ke, v, np.arange(10))
    assert np.allclose(oe[9, 0], v[:, 0].astype(np.float64).mean(0), rtol=2 ** -8, atol=1e-6)


def test_attention_equals_split_and_merge_in_fp64():
    """The fixed-split online softmax (the method's algorithm) reaches the explicit softmax."""
    rng = np.random.default_rng(12)
    L, hd, split, tile = 300, 16, 128, 32
    q = bf16_vals(rng, (L, 1, hd)).astype(np.float64)
    k = bf16_vals(rng, (L, 1, hd)).astype(np.float64)
    v = bf16_vals(rng, (L, 1, hd)).astype(np.float64)
    want = ops.attention(q, k, v, np.arange(L))
    sc = 1 / math.sqrt(hd)
    for p in (0, 63, 127, 128, 299):
        parts = []
        for s0 in range(0, p + 1, split):
            m, l, acc = -np.inf, 0.0, np.zeros(hd)
            for t0 in range(s0, min(s0 + split, p + 1), tile):
                idx = np.arange(t0, min(t0 + tile, p + 1))
                s = (k[idx, 0] @ q[p, 0]) * sc
                mn = max(m, s.max())
                a = math.exp(m - mn) if m > -np.inf else 0.0
                pr = np.exp(s - mn)
                l = l * a + pr.sum()
                acc = acc * a + pr @ v[idx, 0]
                m = mn
            parts.append((m, l, acc))
        M = max(pp[0] for pp in parts)
        Lsum = sum(pp[1] * math.exp(pp[0] - M) for pp in parts)
        O = sum(pp[2] * math.exp(pp[0] - M) for pp in parts)
        assert np.allclose(want[p, 0], O / Lsum, rtol=2 ** -8, atol=1e-6)


# ----------------------------------------------------------------------------- SwiGLU
def test_silu_mul_zeros_and_torch():
    rng = np.random.default_rng(13)
    g = bf16_vals(rng, (7, 33), 3.0)
    u = bf16_vals(rng, (7, 33))
    assert np.all(ops.silu_mul(np.zeros_like(g), u) == 0)
    assert np.all(ops.silu_mul(g, np.zeros_like(u)) == 0)
    want = torch_bf16(TF.silu(torch.from_numpy(g).double()) * torch.from_numpy(u).double()).numpy()
    got = ops.silu_mul(g, u)
    assert np.all(np.abs(got - want) <= 2 ** -7 * np.abs(want) + 1e-30)
    assert np.mean(got == want) > 0.98


# ----------------------------------------------------------------------------- logprob
def test_logprob_normalises_and_matches_log_softmax():
    rng = np.random.default_rng(14)
    V = 1000
    x = (rng.standard_normal((6, V)) * 3).astype(F32)
    all_lp = np.stack([ops.logprob(x, np.full(6, v)) for v in range(V)], axis=1)
    assert np.allclose(np.exp(all_lp).sum(1), 1.0, atol=1e-12)
    ids = rng.integers(0, V, 6)
    want = torch.log_softmax(torch.from_numpy(x).double(), -1).numpy()[np.arange(6), ids]
    assert np.allclose(ops.logprob(x, ids), want, atol=1e-12)


def test_logprob_closed_forms():
    V = 4096
    assert np.allclose(ops.logprob(np.zeros((2, V), F32), [0, 4095]), -math.log(V), atol=1e-12)
    x = np.zeros((1, V), F32)
    x[0, 77] = 100.0
    assert abs(ops.logprob(x, [77])[0]) < 1e-30 + 1e-38 + V * math.exp(-100)
    assert abs(ops.logprob(x, [3])[0] + 100.0) < 1e-9


def test_argmax_ties_go_to_lowest_id():
    x = np.array([[0.0, 2.0, 1.0, 2.0], [5.0, 5.0, 5.0, 5.0], [-1.0, -3.0, -1.0, -2.0]], F32)
    assert ops.argmax_lowest(x).tolist() == [1, 0, 0]


def test_diff_stats_closed_forms():
    a = np.array([-1.5, -0.25, -3.0])
    assert ops.diff_stats(a, a.copy()) == {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}
    s = ops.diff_stats(np.zeros(2), np.full(2, math.log(2.0)))
    assert abs(s["k3"] - (1.0 - math.log(2.0))) < 1e-15
    assert abs(s["max"] - math.log(2.0)) < 1e-15 and s["std"] == 0.0
    # diffs 0, 0, 0, 2: mean 1/2, population std sqrt(3)/2 (the reading: std over the
    # tokens compared, not a sample estimate, which would give 1)
    s = ops.diff_stats(np.zeros(4), np.array([0.0, 0.0, 0.0, 2.0]))
    assert s["max"] == 2.0 and s["mean"] == 0.5
    assert abs(s["std"] - math.sqrt(3.0) / 2.0) < 1e-15
    # k3 per token is r - 1 - log r >= 0 with r = exp(lp_train - lp_rollout): its mean
    # here is (e^2 - 3) / 4
    assert abs(s["k3"] - (math.exp(2.0) - 3.0) / 4.0) < 1e-14


# ----------------------------------------------------------------------------- MoE
def test_route_topk_bruteforce_and_ties():
    rng = np.random.default_rng(15)
    T, E, k = 50, 16, 4
    x = rng.standard_normal((T, E)).astype(F32)
    x[0, 3] = x[0, 9] = x[0, 12] = 10.0               # a three-way tie at the top
    ids, w = moe.route_topk(x, k)
    for t in range(T):
        want = sorted(range(E), key=lambda e: (-float(x[t, e]), e))[:k]
        assert ids[t].tolist() == want
        sel = x[t, want].astype(np.float64)
        p = np.exp(sel - sel.max())
        assert np.allclose(w[t], p / p.sum(), rtol=1e-6)
    assert ids[0, :3].tolist() == [3, 9, 12]
    assert np.allclose(w.sum(1), 1.0, atol=1e-6)
    # heavy ties at the full expert count: only four distinct logit values
    xt = rng.integers(0, 4, (64, 64)).astype(F32)
    idt, _ = moe.route_topk(xt, 8)
    for t in range(64):
        want = sorted(range(64), key=lambda e: (-float(xt[t, e]), e))[:8]
        assert idt[t].tolist() == want


def _ffn_fp64(x, w13, w2):
    F = w2.shape[1]
    xt = torch.from_numpy(x).double()
    g = torch_bf16(xt @ torch.from_numpy(w13[:F]).double().T)
    u = torch_bf16(xt @ torch.from_numpy(w13[F:]).double().T)
    a = torch_bf16(TF.silu(g) * u)
    return torch_bf16(a @ torch.from_numpy(w2).double().T).numpy()


def test_moe_single_expert_equals_dense_ffn():
    rng = np.random.default_rng(16)
    T, E, d, F = 12, 4, 32, 24
    x = bf16_vals(rng, (T, d))
    w13 = bf16_vals(rng, (E, 2 * F, d), 0.3)
    w2 = bf16_vals(rng, (E, d, F), 0.3)
    logits = rng.standard_normal((T, E)).astype(F32)
    out, ids, w = moe.moe_layer(x, logits, w13, w2, k=1)
    assert np.all(w == 1.0)
    for t in range(T):
        want = _ffn_fp64(x[t:t + 1], w13[ids[t, 0]], w2[ids[t, 0]])
        assert np.all(np.abs(out[t] - want[0]) <= 2 ** -7 * np.abs(want[0]) + 1e-6)


def test_moe_identical_experts_equal_one_expert():
    rng = np.random.default_rng(17)
    T, E, d, F = 10, 8, 16, 12
    x = bf16_vals(rng, (T, d))
    w13 = np.repeat(bf16_vals(rng, (1, 2 * F, d), 0.3), E, axis=0)
    w2 = np.repeat(bf16_vals(rng, (1, d, F), 0.3), E, axis=0)
    logits = rng.standard_normal((T, E)).astype(F32)
    out, _, _ = moe.moe_layer(x, logits, w13, w2, k=3)
    want = _ffn_fp64(x, w13[0], w2[0])
    assert np.all(np.abs(out - want) <= 2 ** -6 * np.abs(want) + 1e-6)


def test_moe_bruteforce_tiny():
    rng = np.random.default_rng(18)
    T, E, d, F, k = 5, 4, 6, 3, 2
    x = bf16_vals(rng, (T, d))
    w13 = bf16_vals(rng, (E, 2 * F, d), 0.5)
    w2 = bf16_vals(rng, (E, d, F), 0.5)
    logits = rng.standard_normal((T, E)).astype(F32)
    out, ids, w = moe.moe_layer(x, logits, w13, w2, k)
    for t in range(T):
        acc = np.zeros(d)
        for s in range(k):
            e = ids[t, s]
            y = _ffn_fp64(x[t:t + 1], w13[e], w2[e])[0]
            acc += float(w[t, s]) * y
        assert np.all(np.abs(out[t] - acc) <= 2 ** -7 * np.abs(acc) + 1e-6)


# ----------------------------------------------------------------------------- whole decoder
def _decoder_fp64_torch(wb, shape, tokens):
    """Decoder restated with torch fp64 library ops and torch's bf16 conversion."""
    W = model.weights_to_f32(wb)
    t = lambda a: torch.from_numpy(np.asarray(a)).double()
    hq, hkv, hd, F = shape.n_heads_q, shape.n_heads_kv, shape.head_dim, shape.ffn
    L = len(tokens)
    r = t(W["embed"][np.asarray(tokens)])
    freq = t(10000.0 ** (-np.arange(hd // 2) * 2.0 / hd))
    rot = torch.polar(torch.ones(L, hd // 2, dtype=torch.float64), torch.arange(L).double()[:, None] * freq[None, :])

    def rope(x):
        z = torch.complex(x[..., : hd // 2], x[..., hd // 2:]) * rot[:, None, :]
        return torch_bf16(torch.cat([z.real, z.imag], -1))

    norm = lambda x, g: torch_bf16(TF.rms_norm(x, (x.shape[-1],), t(g), eps=shape.eps))
    x = norm(r, W["layers"][0]["attn_norm"])
    for li, lw in enumerate(W["layers"]):
        qkv = torch_bf16(x @ t(lw["wqkv"]).T)
        q = rope(qkv[:, : hq * hd].reshape(L, hq, hd)).permute(1, 0, 2)
        k = rope(qkv[:, hq * hd:(hq + hkv) * hd].reshape(L, hkv, hd)).permute(1, 0, 2)
        v = qkv[:, (hq + hkv) * hd:].reshape(L, hkv, hd).permute(1, 0, 2)
        k = k.repeat_interleave(hq // hkv, 0)
        v = v.repeat_interleave(hq // hkv, 0)
        a = torch_bf16(TF.scaled_dot_product_attention(q, k, v, is_causal=True)).permute(1, 0, 2).reshape(L, -1)
        r = torch_bf16(r + torch_bf16(a @ t(lw["wo"]).T))
        x = norm(r, lw["ffn_norm"])
        g = torch_bf16(x @ t(lw["w13"][:F]).T)
        u = torch_bf16(x @ t(lw["w13"][F:]).T)
        y = torch_bf16(TF.silu(g) * u)
        r = torch_bf16(r + torch_bf16(y @ t(lw["w2"]).T))
        nxt = W["layers"][li + 1]["attn_norm"] if li + 1 < len(W["layers"]) else W["final_norm"]
        x = norm(r, nxt)
    logits = x @ t(W["lm_head"]).T
    return torch.log_softmax(logits, -1).numpy()


@pytest.mark.parametrize("n_layers,hq,hkv", [(1, 4, 4), (2, 4, 2)])
def test_decoder_matches_fp64_library_restatement(n_layers, hq, hkv):
    shape = DecoderShape(n_layers, 64, hq, hkv, 16, 96, 128)
    wb = make_decoder_weights(shape, seed=19, w_std=0.25, random_gains=True)
    rng = np.random.default_rng(20)
    toks = rng.integers(0, 128, 24)
    W = model.weights_to_f32(wb)
    rows = np.arange(23)
    _, lp = model.score(W, shape, toks, rows, toks[1:])
    ref = _decoder_fp64_torch(wb, shape, toks)[rows, toks[1:]]
    assert np.max(np.abs(lp - ref)) < 2e-2
    assert np.mean(np.abs(lp - ref)) < 4e-3


def test_decoder_is_causal_and_generation_scoring_consistent():
    shape = DecoderShape(2, 32, 2, 1, 16, 48, 64)
    wb = make_decoder_weights(shape, seed=21, w_std=0.3)
    W = model.weights_to_f32(wb)
    rng = np.random.default_rng(22)
    toks = rng.integers(0, 64, 20)
    h1 = model.hidden_states(W, shape, toks)
    toks2 = toks.copy()
    toks2[12:] = (toks2[12:] + 7) % 64
    h2 = model.hidden_states(W, shape, toks2)
    assert np.array_equal(h1[:12], h2[:12])
    assert not np.array_equal(h1[12:], h2[12:])
    gen, lps = model.greedy_generate(W, shape, toks[:8], 5)
    _, lp2, am = model.score_generation(W, shape, toks[:8], gen)
    assert np.array_equal(am, gen)
    assert np.allclose(lp2, lps, atol=0)
