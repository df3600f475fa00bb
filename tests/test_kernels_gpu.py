"""Per-kernel parity with the CPU oracle and bitwise batch invariance, through the C ABI."""
import math

import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from oracle import moe as omoe
from oracle import ops
from synthetic import bits_to_f32, make_moe_layer, normal_bf16, to_bf16_bits
from tests.gpu_util import bf16_close, dev_bf16, host_f32, same_bits

pytestmark = pytest.mark.gpu
F32 = np.float32


def rng_bf16(rng, shape, std=1.0):
    b = normal_bf16(rng, shape, std)
    return b, bits_to_f32(b)


# ---------------------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("rows,d", [(1, 256), (7, 512), (130, 2048), (33, 4096), (5, 520)])
@pytest.mark.parametrize("residual", [False, True])
def test_rmsnorm_parity_and_residual(rows, d, residual):
    rng = np.random.default_rng(rows * d)
    xb, xf = rng_bf16(rng, (rows, d), 2.0)
    rb, rf = rng_bf16(rng, (rows, d))
    gb, gf = rng_bf16(rng, (d,), 0.2)
    gb = normal_bf16(np.random.default_rng(1), (d,), 0.2)
    gf = bits_to_f32(gb) + F32(0)
    x, g = dev_bf16(xb), dev_bf16(gb)
    res = dev_bf16(rb) if residual else None
    y = torch.empty_like(x)
    bi.bi_rmsnorm(x, res, g, y, rows, d, 1e-6)
    want, r_want = ops.rmsnorm(xf, gf, 1e-6, residual=rf if residual else None)
    bf16_close(host_f32(y), want, ulps=1, frac_exact=0.97)
    if residual:
        assert np.array_equal(host_f32(res), r_want)


def test_rmsnorm_rows_do_not_depend_on_batch():
    rng = np.random.default_rng(3)
    d = 2048
    xb, _ = rng_bf16(rng, (300, d))
    g = dev_bf16(normal_bf16(rng, (d,), 1.0))
    x = dev_bf16(xb)
    y = torch.empty_like(x)
    bi.bi_rmsnorm(x, None, g, y, 300, d)
    perm = torch.from_numpy(rng.permutation(300)).cuda()
    xp = x[perm].contiguous()
    yp = torch.empty_like(xp)
    bi.bi_rmsnorm(xp, None, g, yp, 300, d)
    assert same_bits(yp, y[perm])
    for r in (0, 17, 299):
        y1 = torch.empty_like(x[r:r + 1])
        bi.bi_rmsnorm(x[r:r + 1].contiguous(), None, g, y1, 1, d)
        assert same_bits(y1, y[r:r + 1])


# ---------------------------------------------------------------------------- GEMM
# tile widths: 16 below 1M weight elements (SwiGLU: 32 below 2M), 64 below 2M, 128 below 16M (and
# N < 32768), else 256
GEMM_SHAPES = [(1, 64, 64), (5, 1536, 512), (128, 512, 512), (129, 4096, 256), (300, 200, 576), (17, 32000, 512),
               (260, 2816, 512), (131, 3072, 1024), (200, 8192, 2048), (3, 40000, 128), (16, 512, 1408),
               (33, 2048, 768)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_bf16_and_fp32_parity(M, N, K):
    rng = np.random.default_rng(M + N + K)
    ab, af = rng_bf16(rng, (M, K))
    wb, wf = rng_bf16(rng, (N, K), 0.05)
    A, W = dev_bf16(ab), dev_bf16(wb)
    C = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm(A, M, K, W, N, C)
    # fp32 dot products in a different order differ by a small multiple of
    # 2^-24 * sum|a||w|; after rounding both to bf16 the gap is at most one bf16
    # ulp plus that amount.
    absdot = np.abs(af) @ np.abs(wf).T
    bf16_close(host_f32(C), ops.linear(af, wf, "bf16"), ulps=1, frac_exact=0.97, atol=1e-5 * absdot)
    C32 = torch.empty((M, N), dtype=torch.float32, device="cuda")
    bi.bi_gemm(A, M, K, W, N, C32, bi.BI_DTYPE_FP32)
    want = ops.linear(af, wf, "fp32")
    assert np.max(np.abs(host_f32(C32) - want) / (absdot + 1e-30)) < 1e-5


@pytest.mark.parametrize("M,F,K", [(3, 1408, 512), (200, 64, 128), (129, 5632, 256), (70, 4096, 2048)])
def test_gemm_swiglu_epilogue(M, F, K):
    rng = np.random.default_rng(M * F)
    ab, af = rng_bf16(rng, (M, K))
    wb, wf = rng_bf16(rng, (2 * F, K), 0.08)
    C = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm(dev_bf16(ab), M, K, dev_bf16(wb), 2 * F, C, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU)
    want = ops.silu_mul(ops.linear(af, wf[:F]), ops.linear(af, wf[F:]))
    absdot = np.maximum(np.abs(af) @ np.abs(wf[:F]).T, np.abs(af) @ np.abs(wf[F:]).T)
    bf16_close(host_f32(C), want, ulps=2, frac_exact=0.9, atol=2e-2 * absdot * 2.0 ** -7)


@pytest.mark.parametrize("N,K", [(1536, 512), (32000, 512), (512, 1408), (3072, 2048), (8192, 2048), (2048, 768)])
def test_gemm_rows_invariant_to_M_and_order(N, K):
    rng = np.random.default_rng(N)
    ab, _ = rng_bf16(rng, (300, K))
    wb, _ = rng_bf16(rng, (N, K), 0.02)
    A, W = dev_bf16(ab), dev_bf16(wb)
    full = torch.empty((300, N), dtype=torch.float32, device="cuda")
    bi.bi_gemm(A, 300, K, W, N, full, bi.BI_DTYPE_FP32)
    for M in (1, 2, 7, 16, 17, 33, 64, 65, 127, 128, 129, 255):
        part = torch.empty((M, N), dtype=torch.float32, device="cuda")
        off = 300 - M
        bi.bi_gemm(A[off:].contiguous(), M, K, W, N, part, bi.BI_DTYPE_FP32)
        assert same_bits(part, full[off:]), M
    perm = torch.from_numpy(rng.permutation(300)).cuda()
    outp = torch.empty_like(full)
    bi.bi_gemm(A[perm].contiguous(), 300, K, W, N, outp, bi.BI_DTYPE_FP32)
    assert same_bits(outp, full[perm])


@pytest.mark.parametrize("F,K", [(1408, 512), (64, 128), (5632, 2048)])
def test_gemm_swiglu_rows_invariant_to_M_and_order(F, K):
    """The SwiGLU epilogue's 32-, 128- and 256-wide tiles: a row's output bits do not
    depend on how many rows the call has or where the row sits."""
    rng = np.random.default_rng(F + K)
    ab, _ = rng_bf16(rng, (300, K))
    wb, _ = rng_bf16(rng, (2 * F, K), 0.05)
    A, W = dev_bf16(ab), dev_bf16(wb)
    full = torch.empty((300, F), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm(A, 300, K, W, 2 * F, full, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU)
    for M in (1, 16, 17, 40, 64, 129):
        part = torch.empty((M, F), dtype=torch.bfloat16, device="cuda")
        bi.bi_gemm(A[300 - M:].contiguous(), M, K, W, 2 * F, part, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU)
        assert same_bits(part, full[300 - M:]), M
    perm = torch.from_numpy(rng.permutation(300)).cuda()
    outp = torch.empty_like(full)
    bi.bi_gemm(A[perm].contiguous(), 300, K, W, 2 * F, outp, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU)
    assert same_bits(outp, full[perm])


def test_gemm_fast_mode_is_close_but_split():
    """BI_FAST splits K for 17..128 rows (its M-dependent plan; at most 16 rows it
    takes the decode-size schedule like the invariant mode): close to the oracle."""
    rng = np.random.default_rng(9)
    M, N, K = 48, 1536, 512
    ab, af = rng_bf16(rng, (M, K))
    wb, wf = rng_bf16(rng, (N, K), 0.05)
    ws = torch.empty(bi.bi_gemm_workspace_size(M, N, K, 0, bi.BI_FAST), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    C = torch.empty((M, N), dtype=torch.float32, device="cuda")
    bi.bi_gemm(dev_bf16(ab), M, K, dev_bf16(wb), N, C, bi.BI_DTYPE_FP32, 0, bi.BI_FAST, ws)
    want = ops.linear(af, wf, "fp32")
    assert np.max(np.abs(host_f32(C) - want)) < 1e-4


# ---------------------------------------------------------------------------- logprob
@pytest.mark.parametrize("T,V", [(37, 4096), (16, 32000), (3, 129280)])
def test_logprob_gather_parity(T, V):
    rng = np.random.default_rng(T + V)
    x = (rng.standard_normal((T, V)) * 3).astype(F32)
    ids = rng.integers(0, V, T).astype(np.int32)
    xl = torch.from_numpy(x).cuda()
    lp = torch.empty(T, dtype=torch.float32, device="cuda")
    am = torch.empty(T, dtype=torch.int32, device="cuda")
    bi.bi_logprob_gather(xl, torch.from_numpy(ids).cuda(), T, V, lp, am)
    assert np.max(np.abs(lp.cpu().numpy() - ops.logprob(x, ids))) < 5e-5
    assert np.array_equal(am.cpu().numpy(), ops.argmax_lowest(x))
    bi.bi_logprob_gather(xl, None, T, V, lp, am)   # greedy: logprob of the argmax
    assert np.max(np.abs(lp.cpu().numpy() - ops.logprob(x, ops.argmax_lowest(x)))) < 5e-5


def test_logprob_argmax_ties_lowest_id_and_row_invariance():
    V = 32000
    x = np.random.default_rng(5).standard_normal((64, V)).astype(F32)
    x[:, [7, 19000, 31999]] = 9.0
    xl = torch.from_numpy(x).cuda()
    lp = torch.empty(64, dtype=torch.float32, device="cuda")
    am = torch.empty(64, dtype=torch.int32, device="cuda")
    bi.bi_logprob_gather(xl, None, 64, V, lp, am)
    assert (am.cpu().numpy() == 7).all()
    for T in (1, 5, 33):
        lp1 = torch.empty(T, dtype=torch.float32, device="cuda")
        bi.bi_logprob_gather(xl[-T:].contiguous(), None, T, V, lp1)
        assert same_bits(lp1, lp[-T:])


def _fused_head(X, W, ids, mode=bi.BI_INVARIANT):
    T, K = X.shape
    V = W.shape[0]
    lp = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
    am = torch.full((T,), -1, dtype=torch.int32, device="cuda")
    ws = torch.empty(bi.bi_lm_head_logprob_workspace_size(T, V, K, mode), dtype=torch.uint8, device="cuda")
    bi.bi_lm_head_logprob(X, T, K, W, V, ids, lp, am, mode, ws)
    return lp, am


@pytest.mark.parametrize("T,K,V", [(1, 512, 32000), (37, 256, 4096), (130, 512, 32000), (5, 1024, 129280)])
def test_fused_lm_head_logprob_parity_and_row_invariance(T, K, V):
    rng = np.random.default_rng(T * 7 + V)
    xb, xf = rng_bf16(rng, (T, K))
    wb, wf = rng_bf16(rng, (V, K), 0.05)
    ids = rng.integers(0, V, T).astype(np.int32)
    X, W, I = dev_bf16(xb), dev_bf16(wb), torch.from_numpy(ids).cuda()
    lp, am = _fused_head(X, W, I)
    logits = ops.linear(xf, wf, "fp32")
    assert np.max(np.abs(lp.cpu().numpy() - ops.logprob(logits, ids))) < 1e-4
    o_am = ops.argmax_lowest(logits)
    top2 = np.sort(logits, axis=1)[:, -2:]
    clear = (top2[:, 1] - top2[:, 0]) > 1e-4
    assert np.array_equal(am.cpu().numpy()[clear], o_am[clear])
    lpg, amg = _fused_head(X, W, None)                        # greedy
    assert torch.equal(amg, am)
    assert np.max(np.abs(lpg.cpu().numpy() - ops.logprob(logits, amg.cpu().numpy()))) < 1e-4
    for t0 in (0, T // 2, T - 1):                              # rows alone give the same bits
        l1, a1 = _fused_head(X[t0:t0 + 1].contiguous(), W, I[t0:t0 + 1].contiguous())
        assert same_bits(l1, lp[t0:t0 + 1]) and torch.equal(a1, am[t0:t0 + 1])
    lf, _ = _fused_head(X, W, I, bi.BI_FAST)                   # the non-invariant path agrees closely
    assert np.max(np.abs(lf.cpu().numpy() - lp.cpu().numpy())) < 1e-4


@pytest.mark.parametrize("K,V", [(256, 4096), (512, 32000), (256, 1000)])
def test_fused_lm_head_decode_rows_equal_large_calls_on_ties_and_rising_maxima(K, V):
    """Decode-size calls of the fused head (1, 7 and 16 rows) give the bits of a
    40-row call for every row: logits tied exactly (duplicated
    weight rows, within and across vocab tiles) and maxima that rise step after
    step inside a tile (weight rows scaled up column by column), targets on the
    tied and rising columns, and greedy decoding.  V = 1000 ends inside a vocab
    tile (the groups past the last column are skipped)."""
    rng = np.random.default_rng(K + V)
    T = 40
    xb, _ = rng_bf16(rng, (T, K))
    wb, wf = rng_bf16(rng, (V, K), 0.05)
    wf = wf.copy()
    # exact ties: column 3 equals column 1 (one tile), column 200 equals column 1 (another tile)
    wf[3] = wf[1]
    wf[200] = wf[1]
    # rising maxima: columns 64..127 of the second tile scaled up 1.05x per column
    wf[64:128] = wf[1][None, :] * (1.05 ** np.arange(1, 65))[:, None]
    wb = to_bf16_bits(wf)
    ids = rng.integers(0, V, T).astype(np.int32)
    ids[:8] = [1, 3, 200, 64, 127, 100, V - 1, 0]
    X, W, I = dev_bf16(xb), dev_bf16(wb), torch.from_numpy(ids).cuda()
    lp, am = _fused_head(X, W, I)
    lpg, amg = _fused_head(X, W, None)
    for M in (1, 7, 16):
        for t0 in (0, 13, T - M):
            sl = slice(t0, t0 + M)
            l1, a1 = _fused_head(X[sl].contiguous(), W, I[sl].contiguous())
            assert same_bits(l1, lp[sl]) and torch.equal(a1, am[sl]), (M, t0)
            l2, a2 = _fused_head(X[sl].contiguous(), W, None)
            assert same_bits(l2, lpg[sl]) and torch.equal(a2, amg[sl]), (M, t0)
    assert bi.bi_device_status() == 0


# ---------------------------------------------------------------------------- RoPE + attention
def _paged_setup(seq_lens, Hq, Hkv, hd, rng, n_blocks_extra=3):
    max_blk = max(math.ceil(n / 64) for n in seq_lens)
    n_blocks = len(seq_lens) * max_blk + n_blocks_extra
    perm = rng.permutation(n_blocks)[: len(seq_lens) * max_blk].astype(np.int32)
    bt = torch.from_numpy(perm.reshape(len(seq_lens), max_blk)).cuda()
    kc = torch.full((n_blocks, Hkv, 64, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full((n_blocks, Hkv, 64, hd), float("nan"), dtype=torch.bfloat16, device="cuda")
    return bt, kc, vc, max_blk, n_blocks


def _pieces(pieces):
    """pieces: list of (seq, pos0, n) -> device metadata arrays."""
    seq = torch.tensor([p[0] for p in pieces], dtype=torch.int32, device="cuda")
    row0 = torch.tensor(np.concatenate([[0], np.cumsum([p[2] for p in pieces])]), dtype=torch.int32, device="cuda")
    pos0 = torch.tensor([p[1] for p in pieces], dtype=torch.int32, device="cuda")
    return seq, row0, pos0


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 8, 64), (16, 4, 128), (4, 1, 64)])
def test_rope_kv_write_and_attention_prefill_parity(Hq, Hkv, hd):
    rng = np.random.default_rng(Hq * hd)
    seq_lens = [70, 600, 1100]
    bt, kc, vc, max_blk, n_blocks = _paged_setup(seq_lens, Hq, Hkv, hd, rng)
    max_pos = 2048
    table = torch.empty((max_pos, hd), dtype=torch.float32, device="cuda")
    bi.bi_rope_table(table, max_pos, hd, 10000.0)
    nq = (Hq + 2 * Hkv) * hd
    T = sum(seq_lens)
    qkvb, qkvf = rng_bf16(rng, (T, nq))
    seq, row0, pos0 = _pieces([(b, 0, n) for b, n in enumerate(seq_lens)])
    q = torch.empty((T, Hq, hd), dtype=torch.bfloat16, device="cuda")
    bi.bi_rope_kv_write(dev_bf16(qkvb), T, seq, row0, pos0, len(seq_lens), max(seq_lens), Hq, Hkv, hd, table, max_pos,
                        bt, max_blk, n_blocks, q, kc, vc)
    out = torch.empty((T, Hq * hd), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bi.bi_attention_workspace_size(T, Hq, hd, max(seq_lens), 512), dtype=torch.uint8, device="cuda")
    bi.bi_attention(q, T, seq, row0, pos0, len(seq_lens), max(seq_lens), Hq, Hkv, hd, kc, vc, bt, max_blk,
                    kc.shape[0], max(seq_lens), 512, 1.0 / math.sqrt(hd), ws, out)
    got_q, got_o = host_f32(q), host_f32(out)
    r0 = 0
    for b, n in enumerate(seq_lens):
        f = qkvf[r0:r0 + n]
        pos = np.arange(n)
        qo = ops.rope(f[:, : Hq * hd].reshape(n, Hq, hd), pos)
        ko = ops.rope(f[:, Hq * hd:(Hq + Hkv) * hd].reshape(n, Hkv, hd), pos)
        vo = f[:, (Hq + Hkv) * hd:].reshape(n, Hkv, hd)
        bf16_close(got_q[r0:r0 + n], qo, ulps=1, frac_exact=0.99)
        # cache contents at the sequence's blocks
        blocks = bt[b].cpu().numpy()
        kg = host_f32(kc)[blocks].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n]
        vg = host_f32(vc)[blocks].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n]
        bf16_close(kg, ko, ulps=1, frac_exact=0.99)
        assert np.array_equal(vg, vo)
        want = ops.attention(qo, ko, vo, pos).reshape(n, Hq * hd)
        err = np.abs(got_o[r0:r0 + n] - want)
        assert err.max() < 2e-2 and err.mean() < 2e-3, (err.max(), err.mean())
        r0 += n


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 8, 64), (16, 4, 128)])
def test_attention_decode_rows_equal_prefill_rows_bitwise(Hq, Hkv, hd):
    """A decode call (one token per sequence) reproduces the prefill rows exactly,
    and so does any chunking of the prefill."""
    rng = np.random.default_rng(11 + hd)
    seq_lens = [1100, 513, 64, 1]
    bt, kc, vc, max_blk, n_blocks = _paged_setup(seq_lens, Hq, Hkv, hd, rng)
    max_pos = 2048
    table = torch.empty((max_pos, hd), dtype=torch.float32, device="cuda")
    bi.bi_rope_table(table, max_pos, hd, 10000.0)
    nq = (Hq + 2 * Hkv) * hd
    T = sum(seq_lens)
    qkv = dev_bf16(normal_bf16(rng, (T, nq), 1.0))
    scale = 1.0 / math.sqrt(hd)

    def run(pieces, rows_qkv, max_ctx, mode=bi.BI_INVARIANT):
        seq, row0, pos0 = _pieces(pieces)
        Tn = rows_qkv.shape[0]
        mq = max(p[2] for p in pieces)
        q = torch.empty((Tn, Hq, hd), dtype=torch.bfloat16, device="cuda")
        bi.bi_rope_kv_write(rows_qkv, Tn, seq, row0, pos0, len(pieces), mq, Hq, Hkv, hd, table, max_pos, bt, max_blk,
                            n_blocks, q, kc, vc)
        out = torch.empty((Tn, Hq * hd), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bi.bi_attention_workspace_size(Tn, Hq, hd, max_ctx, 512), dtype=torch.uint8, device="cuda")
        bi.bi_attention(q, Tn, seq, row0, pos0, len(pieces), mq, Hq, Hkv, hd, kc, vc, bt, max_blk, kc.shape[0], max_ctx,
                        512, scale, ws, out, mode)
        return out

    offs = np.concatenate([[0], np.cumsum(seq_lens)])
    full = run([(b, 0, n) for b, n in enumerate(seq_lens)], qkv, max(seq_lens))
    # chunked prefill: chunks of 97 then of 64
    for ch in (97, 64, 512):
        outs = []
        for b, n in enumerate(seq_lens):
            for s0 in range(0, n, ch):
                e = min(n, s0 + ch)
                outs.append((offs[b] + s0, run([(b, s0, e - s0)], qkv[offs[b] + s0: offs[b] + e].contiguous(),
                                               max(seq_lens))))
        for r, o in outs:
            assert same_bits(o, full[r:r + o.shape[0]]), ch
    # decode: every sequence's rows at a few positions, as one batch of single tokens
    for pos in (0, 63, 64, 511, 512, 1099):
        pcs, rows = [], []
        for b, n in enumerate(seq_lens):
            if pos < n:
                pcs.append((b, pos, 1))
                rows.append(offs[b] + pos)
        if not pcs:
            continue
        # max_ctx 2048: one CTA per (sequence, kv head, split); 8192: the persistent schedule
        for max_ctx in (2048, 8192):
            o = run(pcs, qkv[torch.tensor(rows, device="cuda")].contiguous(), max_ctx)
            assert same_bits(o, full[torch.tensor(rows, device="cuda")]), (pos, max_ctx)


@pytest.mark.parametrize("Hq,Hkv,hd,B", [(8, 8, 64, 300), (16, 4, 128, 200), (8, 1, 64, 1100)])
def test_attention_decode_schedules_agree(Hq, Hkv, hd, B):
    """Decode rows are bitwise the same whichever decode schedule runs: per-CTA
    (max_ctx 2048 = 4 splits) or persistent with TMA page streaming (max_ctx
    16384; more than 1024 sequences fall back to per-CTA).  Cache slots after
    each sequence's last position hold NaN, which must never reach the output."""
    rng = np.random.default_rng(B * 3 + hd)
    ctx = rng.integers(1, 2049, B)
    max_blk = 32
    n_blocks = B * max_blk
    bt = torch.from_numpy(rng.permutation(n_blocks).astype(np.int32).reshape(B, max_blk)).cuda()
    kc = (0.5 * torch.randn((n_blocks, Hkv, 64, hd), device="cuda")).to(torch.bfloat16)
    vc = (0.5 * torch.randn((n_blocks, Hkv, 64, hd), device="cuda")).to(torch.bfloat16)
    stale = np.zeros((n_blocks, 64), dtype=bool)
    tab = bt.cpu().numpy()
    for b in range(B):
        last = (ctx[b] - 1) // 64
        stale[tab[b, last], ctx[b] - last * 64:] = True
        stale[tab[b, last + 1:]] = True
    m = torch.from_numpy(stale).cuda()
    kc.permute(0, 2, 1, 3)[m] = float("nan")
    vc.permute(0, 2, 1, 3)[m] = float("nan")
    q = (0.5 * torch.randn((B, Hq, hd), device="cuda")).to(torch.bfloat16)
    seq = torch.arange(B, dtype=torch.int32, device="cuda")
    row0 = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    pos0 = torch.from_numpy((ctx - 1).astype(np.int32)).cuda()
    outs = []
    for max_ctx in (2048, 16384):
        out = torch.empty((B, Hq * hd), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bi.bi_attention_workspace_size(B, Hq, hd, max_ctx, 512), dtype=torch.uint8, device="cuda")
        bi.bi_attention(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, kc, vc, bt, max_blk, n_blocks, max_ctx, 512,
                        hd ** -0.5, ws, out)
        outs.append(out)
    assert bi.bi_device_status() == 0
    assert not torch.isnan(outs[0].float()).any()
    assert same_bits(outs[1], outs[0])


@pytest.mark.parametrize("Hq,Hkv,hd,B", [(8, 8, 64, 16), (8, 2, 64, 300), (4, 1, 64, 37), (16, 4, 128, 40)])
def test_attention_decode_two_split_schedule(Hq, Hkv, hd, B):
    """Decode calls whose contexts fit two splits (max_ctx <= 1024) take, at hd 64,
    the schedule that covers both splits in one CTA and merges them there.  Its
    rows equal, bit for bit, those of the per-split schedule (max_ctx 2048) and of
    the persistent one (max_ctx 16384), and match the oracle's explicit softmax
    (rows before, at and after the split boundary).  Slots after each sequence's
    last position hold NaN."""
    rng = np.random.default_rng(B + 5 * hd + Hkv)
    ctx = rng.integers(1, 1025, B)
    ctx[: min(B, 4)] = [1, 512, 513, 1024][: min(B, 4)]
    max_blk = 16
    n_blocks = B * max_blk
    bt = torch.from_numpy(rng.permutation(n_blocks).astype(np.int32).reshape(B, max_blk)).cuda()
    kb = normal_bf16(rng, (n_blocks, Hkv, 64, hd), 0.5)
    vb = normal_bf16(rng, (n_blocks, Hkv, 64, hd), 0.5)
    kc, vc = dev_bf16(kb), dev_bf16(vb)
    stale = np.zeros((n_blocks, 64), dtype=bool)
    tab = bt.cpu().numpy()
    for b in range(B):
        last = (ctx[b] - 1) // 64
        stale[tab[b, last], ctx[b] - last * 64:] = True
        stale[tab[b, last + 1:]] = True
    m = torch.from_numpy(stale).cuda()
    kc.permute(0, 2, 1, 3)[m] = float("nan")
    vc.permute(0, 2, 1, 3)[m] = float("nan")
    qb = normal_bf16(rng, (B, Hq, hd), 0.5)
    q = dev_bf16(qb)
    seq = torch.arange(B, dtype=torch.int32, device="cuda")
    row0 = torch.arange(B + 1, dtype=torch.int32, device="cuda")
    pos0 = torch.from_numpy((ctx - 1).astype(np.int32)).cuda()
    outs = []
    for max_ctx in (1024, 2048, 16384):
        out = torch.empty((B, Hq * hd), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bi.bi_attention_workspace_size(B, Hq, hd, max_ctx, 512), dtype=torch.uint8, device="cuda")
        bi.bi_attention(q, B, seq, row0, pos0, B, 1, Hq, Hkv, hd, kc, vc, bt, max_blk, n_blocks, max_ctx, 512,
                        hd ** -0.5, ws, out)
        outs.append(out)
    assert bi.bi_device_status() == 0
    assert not torch.isnan(outs[0].float()).any()
    assert same_bits(outs[1], outs[0]) and same_bits(outs[2], outs[0])
    got = host_f32(outs[0]).reshape(B, Hq, hd)
    kf, vf = bits_to_f32(kb), bits_to_f32(vb)
    for b in range(min(B, 4)):
        n = int(ctx[b])
        blocks = tab[b, : (n + 63) // 64]
        k = kf[blocks].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n]
        v = vf[blocks].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n]
        want = ops.attention(bits_to_f32(qb[b:b + 1]), k, v, np.array([n - 1]))
        err = np.abs(got[b] - want[0])
        assert err.max() < 2e-2 and err.mean() < 2e-3, (b, n, err.max(), err.mean())


# ---------------------------------------------------------------------------- MoE
def _moe_dev(T, d, F, E, seed):
    inp = make_moe_layer(T, d, F, E, 0.05, seed)
    return inp, dev_bf16(inp["x"]), torch.from_numpy(inp["router_logits"]).cuda(), dev_bf16(inp["w13"]), \
        dev_bf16(inp["w2"])


def test_moe_route_topk_matches_oracle_and_ties():
    rng = np.random.default_rng(2)
    T, E, k = 500, 64, 8
    x = rng.standard_normal((T, E)).astype(F32)
    x[:50] = np.round(x[:50])   # many exact ties
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    bi.bi_moe_route_topk(torch.from_numpy(x).cuda(), T, E, k, ids, w)
    oi, ow = omoe.route_topk(x, k)
    assert np.array_equal(ids.cpu().numpy(), oi)
    assert np.max(np.abs(w.cpu().numpy() - ow)) < 1e-6


def _stable_layout(ids, E, cap=0):
    """Host reference: the rank of each (token, slot) pair among the earlier pairs of its
    expert (a stable counting sort), then its row in the contiguous layout (expert ranges
    padded to 128, in expert order) or the masked one (cap rows per expert, -1 beyond)."""
    ids = np.asarray(ids).ravel()
    seen = np.zeros(E, np.int64)
    rank = np.empty(len(ids), np.int64)
    for i, e in enumerate(ids):
        rank[i] = seen[e]
        seen[e] += 1
    if cap:
        rows = np.where(rank < cap, ids * cap + rank, -1)
        return rows, None, np.arange(E * cap // 128) // (cap // 128)
    off = np.concatenate([[0], np.cumsum((seen + 127) // 128 * 128)])
    return off[ids] + rank, off, off


@pytest.mark.parametrize("case", ["uniform", "skewed", "one_expert", "wide"])
def test_moe_permute_is_a_stable_counting_sort(case):
    """bi_moe_permute / bi_moe_permute_masked against a host stable counting sort, bit for bit:
    ragged pair counts (not a multiple of the 1024-pair chunk), empty experts, one expert
    taking every pair, E up to 1000, and masked capacity overflow (dropped and reported)."""
    rng = np.random.default_rng({"uniform": 1, "skewed": 2, "one_expert": 3, "wide": 4}[case])
    T, k, E = {"uniform": (4096, 8, 64), "skewed": (777, 8, 64), "one_expert": (300, 1, 64),
               "wide": (2500, 4, 1000)}[case]
    if case == "skewed":
        ids = np.minimum(rng.geometric(0.15, (T, k)) - 1, E - 1)           # many empty experts
    elif case == "one_expert":
        ids = np.full((T, k), 17)
    else:
        ids = rng.integers(0, E, (T, k))
    ids = ids.astype(np.int32)
    d_ids = torch.from_numpy(ids).cuda()
    max_rows = 128 * math.ceil((T * k + 127 * E) / 128)
    ros = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
    tiles = torch.full((max_rows // 128,), -7, dtype=torch.int32, device="cuda")
    offs = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
    pws = torch.empty(bi.bi_moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    bi.bi_moe_permute(d_ids, T, k, E, max_rows, ros, tiles, offs, pws)
    rows, off, _ = _stable_layout(ids, E)
    assert np.array_equal(ros.cpu().numpy(), rows)
    assert np.array_equal(offs.cpu().numpy(), off)
    t_start = np.arange(max_rows // 128) * 128
    owner = np.where(t_start < off[-1], np.searchsorted(off[1:], t_start, side="right"), -1)
    assert np.array_equal(tiles.cpu().numpy(), owner)
    assert bi.bi_device_status() == 0
    # masked layout; the smallest capacity that holds every pair first, then one that drops some
    need = int(np.bincount(ids.ravel(), minlength=E).max())
    for cap, overflow in ((128 * math.ceil(need / 128), False), (128, need > 128)):
        ros_m = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
        tiles_m = torch.full((E * cap // 128,), -7, dtype=torch.int32, device="cuda")
        bi.bi_moe_permute_masked(d_ids, T, k, E, cap, ros_m, tiles_m, pws)
        rows_m, _, owner_m = _stable_layout(ids, E, cap)
        assert np.array_equal(ros_m.cpu().numpy(), rows_m)
        assert np.array_equal(tiles_m.cpu().numpy(), owner_m)
        st = bi.bi_device_status()                     # reading it also clears it
        assert (st == bi.BI_ERR_DEVICE_CHECK) == overflow, st


@pytest.mark.parametrize("T", [1, 37, 512])
def test_moe_layer_parity(T):
    d, F, E, k = 256, 128, 16, 4
    inp, x, lg, w13, w2 = _moe_dev(T, d, F, E, seed=T)
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bi.bi_moe_layer_workspace_size(T, d, E, k, F), dtype=torch.uint8, device="cuda")
    bi.bi_moe_layer(x, lg, T, d, E, k, F, w13, w2, out, bi.BI_INVARIANT, ws)
    want, _, _ = omoe.moe_layer(bits_to_f32(inp["x"]), inp["router_logits"], bits_to_f32(inp["w13"]),
                                bits_to_f32(inp["w2"]), k)
    got = host_f32(out)
    err = np.abs(got - want)
    assert np.all(err <= 2 * 2.0 ** -7 * np.abs(want) + 2e-3), err.max()


def test_moe_rows_invariant_to_batching_and_layout():
    T, d, F, E, k = 600, 256, 128, 16, 4
    inp, x, lg, w13, w2 = _moe_dev(T, d, F, E, seed=77)

    def layer(xs, ls):
        n = xs.shape[0]
        out = torch.empty((n, d), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bi.bi_moe_layer_workspace_size(n, d, E, k, F), dtype=torch.uint8, device="cuda")
        bi.bi_moe_layer(xs, ls, n, d, E, k, F, w13, w2, out, bi.BI_INVARIANT, ws)
        return out

    full = layer(x, lg)
    rng = np.random.default_rng(0)
    perm = torch.from_numpy(rng.permutation(T)).cuda()
    assert same_bits(layer(x[perm].contiguous(), lg[perm].contiguous()), full[perm])
    for a, b in ((0, 1), (5, 200), (300, 600)):
        assert same_bits(layer(x[a:b].contiguous(), lg[a:b].contiguous()), full[a:b])
    # masked layout (fixed capacity per expert) gives the same rows as the contiguous one
    ids = torch.empty((T, k), dtype=torch.int32, device="cuda")
    w = torch.empty((T, k), dtype=torch.float32, device="cuda")
    bi.bi_moe_route_topk(lg, T, E, k, ids, w)
    cap = 128 * math.ceil(T * k / E / 128 + 2)
    ros = torch.empty(T * k, dtype=torch.int32, device="cuda")
    tiles = torch.empty(E * cap // 128, dtype=torch.int32, device="cuda")
    pws = torch.empty(bi.bi_moe_permute_workspace_size(T, k, E), dtype=torch.uint8, device="cuda")
    bi.bi_moe_permute_masked(ids, T, k, E, cap, ros, tiles, pws)
    xp = torch.zeros((E * cap, d), dtype=torch.bfloat16, device="cuda")
    bi.bi_moe_gather(x, ros, T, k, d, xp)
    act = torch.empty((E * cap, F), dtype=torch.bfloat16, device="cuda")
    bi.bi_grouped_gemm(xp, E * cap, d, w13, E, 2 * F, tiles, act, bi.BI_DTYPE_BF16, bi.BI_EPI_SWIGLU)
    y = torch.empty((E * cap, d), dtype=torch.bfloat16, device="cuda")
    bi.bi_grouped_gemm(act, E * cap, F, w2, E, d, tiles, y)
    out = torch.empty((T, d), dtype=torch.bfloat16, device="cuda")
    bi.bi_moe_combine(y, ros, w, T, k, d, out)
    assert same_bits(out, full)


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 8, 64), (16, 4, 128)])
def test_fused_qkv_rope_kv_write_equals_gemm_then_rope(Hq, Hkv, hd):
    """The QKV GEMM with RoPE + paged K/V write in its epilogue gives the same q
    and cache bits as bi_gemm followed by bi_rope_kv_write."""
    rng = np.random.default_rng(Hq + hd)
    seq_lens = [130, 1, 77]
    T, K = sum(seq_lens), 512
    N = (Hq + 2 * Hkv) * hd
    xb, _ = rng_bf16(rng, (T, K))
    wb, _ = rng_bf16(rng, (N, K), 0.05)
    X, W = dev_bf16(xb), dev_bf16(wb)
    max_pos = 1024
    table = torch.empty((max_pos, hd), dtype=torch.float32, device="cuda")
    bi.bi_rope_table(table, max_pos, hd, 10000.0)
    starts = [3, 0, 200]                      # rows sit at positions start + i
    bt, kc1, vc1, max_blk, n_blocks = _paged_setup([s + n for s, n in zip(starts, seq_lens)], Hq, Hkv, hd, rng)
    kc1.zero_()
    vc1.zero_()
    kc2, vc2 = torch.zeros_like(kc1), torch.zeros_like(vc1)
    seq, row0, pos0 = _pieces([(b, starts[b], n) for b, n in enumerate(seq_lens)])
    qkv = torch.empty((T, N), dtype=torch.bfloat16, device="cuda")
    bi.bi_gemm(X, T, K, W, N, qkv)
    q1 = torch.empty((T, Hq, hd), dtype=torch.bfloat16, device="cuda")
    bi.bi_rope_kv_write(qkv, T, seq, row0, pos0, len(seq_lens), max(seq_lens), Hq, Hkv, hd, table, max_pos, bt,
                        max_blk, n_blocks, q1, kc1, vc1)
    row_seq = torch.tensor(np.repeat(np.arange(len(seq_lens)), seq_lens), dtype=torch.int32, device="cuda")
    row_pos = torch.tensor(np.concatenate([starts[b] + np.arange(n) for b, n in enumerate(seq_lens)]),
                           dtype=torch.int32, device="cuda")
    q2 = torch.empty_like(q1)
    bi.bi_qkv_rope_kv_write(X, T, K, W, Hq, Hkv, hd, row_seq, row_pos, table, max_pos, bt, max_blk, n_blocks, q2,
                            kc2, vc2)
    assert same_bits(q2, q1)
    assert same_bits(kc2, kc1) and same_bits(vc2, vc1)
    assert bi.bi_device_status() == 0


@pytest.mark.parametrize("Hq,Hkv,hd,K", [(8, 8, 64, 512), (16, 4, 128, 512), (16, 4, 128, 2048)])
def test_fused_qkv_rope_rows_invariant_to_M(Hq, Hkv, hd, K):
    """The fused QKV + RoPE + paged K/V write: a decode-size call (M <= 16 rows)
    writes the same q and cache bits for its rows as a 300-row call, whichever
    schedule each call takes."""
    rng = np.random.default_rng(Hq * K + hd)
    seq_lens = [130, 1, 77, 92]
    T = sum(seq_lens)
    N = (Hq + 2 * Hkv) * hd
    xb, _ = rng_bf16(rng, (T, K))
    wb, _ = rng_bf16(rng, (N, K), 0.05)
    X, W = dev_bf16(xb), dev_bf16(wb)
    max_pos = 1024
    table = torch.empty((max_pos, hd), dtype=torch.float32, device="cuda")
    bi.bi_rope_table(table, max_pos, hd, 10000.0)
    starts = [3, 0, 200, 64]
    bt, kc, vc, max_blk, n_blocks = _paged_setup([s + n for s, n in zip(starts, seq_lens)], Hq, Hkv, hd, rng)
    kc.zero_()
    vc.zero_()
    seqs = np.repeat(np.arange(len(seq_lens)), seq_lens).astype(np.int32)
    poss = np.concatenate([starts[b] + np.arange(n) for b, n in enumerate(seq_lens)]).astype(np.int32)
    row_seq, row_pos = torch.from_numpy(seqs).cuda(), torch.from_numpy(poss).cuda()
    q = torch.empty((T, Hq, hd), dtype=torch.bfloat16, device="cuda")
    bi.bi_qkv_rope_kv_write(X, T, K, W, Hq, Hkv, hd, row_seq, row_pos, table, max_pos, bt, max_blk, n_blocks, q,
                            kc, vc)
    btc = bt.cpu().numpy()
    for M in (1, 5, 16, 17, 40, 64):
        idx = np.sort(rng.choice(T, M, replace=False))
        kp, vp = torch.zeros_like(kc), torch.zeros_like(vc)
        qp = torch.empty((M, Hq, hd), dtype=torch.bfloat16, device="cuda")
        it = torch.from_numpy(idx).cuda()
        bi.bi_qkv_rope_kv_write(X[it].contiguous(), M, K, W, Hq, Hkv, hd, row_seq[it].contiguous(),
                                row_pos[it].contiguous(), table, max_pos, bt, max_blk, n_blocks, qp, kp, vp)
        assert same_bits(qp, q[it]), M
        blk = torch.from_numpy(btc[seqs[idx], poss[idx] // 64].astype(np.int64)).cuda()
        slot = torch.from_numpy((poss[idx] % 64).astype(np.int64)).cuda()
        assert same_bits(kp[blk, :, slot], kc[blk, :, slot]) and same_bits(vp[blk, :, slot], vc[blk, :, slot]), M
        written = torch.zeros(kp.shape[0], kp.shape[2], dtype=torch.bool, device="cuda")
        written[blk, slot] = True
        assert not kp.permute(0, 2, 1, 3)[~written].any() and not vp.permute(0, 2, 1, 3)[~written].any(), M
    assert bi.bi_device_status() == 0
