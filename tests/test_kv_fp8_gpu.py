"""FP8 KV cache ([Article] §4.2) through the C ABI: the quantising write and the
dequantise-and-gather read are bit-exact against the oracle, and attention over the
FP8 cache gives the same bits to a decode row and to its prefill row (one read path),
within the bf16 attention tolerance of the oracle on the dequantised history.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own."""
import math

import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from oracle import fp8 as ofp8
from oracle import ops
from synthetic import bits_to_f32, normal_bf16
from tests.gpu_util import dev_bf16, host_f32, same_bits

pytestmark = pytest.mark.gpu


class Fp8Cache:
    def __init__(self, lens, Hkv, hd, rng):
        self.max_blk = max(math.ceil(n / 64) for n in lens)
        self.n_blocks = len(lens) * self.max_blk + 2
        perm = rng.permutation(self.n_blocks)[: len(lens) * self.max_blk].astype(np.int32)
        self.bt = torch.from_numpy(perm.reshape(len(lens), self.max_blk)).cuda()
        self.k8 = torch.full((self.n_blocks, Hkv, 64, hd), 0x7F, dtype=torch.uint8, device="cuda")   # NaN codes
        self.v8 = torch.full_like(self.k8, 0x7F)
        self.ks = torch.full((self.n_blocks, Hkv, 64), float("nan"), device="cuda")
        self.vs = torch.full_like(self.ks, float("nan"))
        self.Hkv, self.hd = Hkv, hd

    def write(self, pieces, kb, vb):
        seq, row0, pos0 = _pieces(pieces)
        T = kb.shape[0]
        bi.bi_kv_fp8_write(dev_bf16(kb), dev_bf16(vb), T, seq, row0, pos0, len(pieces), max(p[2] for p in pieces),
                           self.Hkv, self.hd, self.bt, self.max_blk, self.n_blocks, self.k8, self.v8, self.ks,
                           self.vs)

    def attend(self, pieces, qb, Hq, max_ctx):
        """Gather the pieces' history into a bf16 workspace, then bi_attention over it."""
        seq, row0, pos0 = _pieces(pieces)
        P = len(pieces)
        kw = torch.empty((P * self.max_blk, self.Hkv, 64, self.hd), dtype=torch.bfloat16, device="cuda")
        vw = torch.empty_like(kw)
        wbt = torch.empty((P, self.max_blk), dtype=torch.int32, device="cuda")
        bi.bi_kv_fp8_gather(self.k8, self.v8, self.ks, self.vs, self.n_blocks, seq, row0, pos0, P, self.Hkv, self.hd,
                            self.bt, self.max_blk, kw, vw, wbt)
        T = qb.shape[0]
        out = torch.empty((T, Hq * self.hd), dtype=torch.bfloat16, device="cuda")
        ws = torch.empty(bi.bi_attention_workspace_size(T, Hq, self.hd, max_ctx, 512), dtype=torch.uint8,
                         device="cuda")
        ident = torch.arange(P, dtype=torch.int32, device="cuda")
        bi.bi_attention(dev_bf16(qb), T, ident, row0, pos0, P, max(p[2] for p in pieces), Hq, self.Hkv, self.hd, kw,
                        vw, wbt, self.max_blk, P * self.max_blk, max_ctx, 512, 1.0 / math.sqrt(self.hd), ws, out)
        return out, kw, vw, wbt

    def attend_direct(self, pieces, qb, Hq, max_ctx, quant=False, mode=0):
        """bi_attention_fp8 over the FP8 pages themselves; with quant also the
        quantised output rows.  Returns (out, codes, scales)."""
        seq, row0, pos0 = _pieces(pieces)
        P = len(pieces)
        T = qb.shape[0]
        out = torch.empty((T, Hq * self.hd), dtype=torch.bfloat16, device="cuda")
        oq = torch.empty((T, Hq * self.hd), dtype=torch.uint8, device="cuda") if quant else None
        osc = torch.empty((T, Hq * self.hd // 128), dtype=torch.float32, device="cuda") if quant else None
        ws = torch.empty(bi.bi_attention_workspace_size(T, Hq, self.hd, max_ctx, 512), dtype=torch.uint8,
                         device="cuda")
        bi.bi_attention_fp8(dev_bf16(qb), T, seq, row0, pos0, P, max(p[2] for p in pieces), Hq, self.Hkv, self.hd,
                            self.k8, self.v8, self.ks, self.vs, self.bt, self.max_blk, self.n_blocks, max_ctx, 512,
                            1.0 / math.sqrt(self.hd), ws, out, oq, osc, mode)
        return out, oq, osc


def _pieces(pieces):
    seq = torch.tensor([p[0] for p in pieces], dtype=torch.int32, device="cuda")
    row0 = torch.tensor(np.concatenate([[0], np.cumsum([p[2] for p in pieces])]), dtype=torch.int32, device="cuda")
    pos0 = torch.tensor([p[1] for p in pieces], dtype=torch.int32, device="cuda")
    return seq, row0, pos0


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 8, 64), (16, 4, 128)])
def test_fp8_cache_write_gather_bitexact_and_attention(Hq, Hkv, hd):
    rng = np.random.default_rng(Hq + hd)
    lens = [300, 1, 129, 700]
    T = sum(lens)
    kb, vb = normal_bf16(rng, (T, Hkv, hd), 1.0), normal_bf16(rng, (T, Hkv, hd), 1.0)
    qb = normal_bf16(rng, (T, Hq, hd), 1.0)
    c = Fp8Cache(lens, Hkv, hd, rng)
    c.write([(b, 0, n) for b, n in enumerate(lens)], kb, vb)
    pieces = [(b, 0, n) for b, n in enumerate(lens)]
    out, kw, vw, wbt = c.attend(pieces, qb, Hq, max(lens))
    k8, ks, v8, vs = c.k8.cpu().numpy(), c.ks.cpu().numpy(), c.v8.cpu().numpy(), c.vs.cpu().numpy()
    kwf, vwf, wb = host_f32(kw), host_f32(vw), wbt.cpu().numpy()
    offs = np.concatenate([[0], np.cumsum(lens)])
    got = host_f32(out)
    for b, n in enumerate(lens):
        kf, vf = bits_to_f32(kb[offs[b]:offs[b] + n]), bits_to_f32(vb[offs[b]:offs[b] + n])
        qk, sk = ofp8.quantize_blocks(kf.reshape(-1, hd), 1, block_cols=hd)
        qv, sv = ofp8.quantize_blocks(vf.reshape(-1, hd), 1, block_cols=hd)
        blocks = c.bt[b].cpu().numpy()
        # the cache's codes and scales at the sequence's slots
        gk = k8[blocks].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n].reshape(-1, hd)
        gv = v8[blocks].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n].reshape(-1, hd)
        assert np.array_equal(gk, qk) and np.array_equal(gv, qv)
        assert np.array_equal(ks[blocks].transpose(0, 2, 1).reshape(-1, Hkv)[:n].reshape(-1), sk[:, 0])
        assert np.array_equal(vs[blocks].transpose(0, 2, 1).reshape(-1, Hkv)[:n].reshape(-1), sv[:, 0])
        # the gathered workspace holds exactly the dequantised history
        kd = ofp8.dequantize_blocks(qk, sk, 1, block_cols=hd).reshape(n, Hkv, hd)
        vd = ofp8.dequantize_blocks(qv, sv, 1, block_cols=hd).reshape(n, Hkv, hd)
        pages = wb[b][wb[b] >= 0]
        assert np.array_equal(pages, b * c.max_blk + np.arange(len(pages)))
        assert np.array_equal(kwf[pages].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n], kd)
        assert np.array_equal(vwf[pages].transpose(0, 2, 1, 3).reshape(-1, Hkv, hd)[:n], vd)
        # attention over the FP8 history vs the explicit-softmax oracle on the dequantised K/V
        want = ops.attention(bits_to_f32(qb[offs[b]:offs[b] + n]), kd, vd, np.arange(n)).reshape(n, Hq * hd)
        err = np.abs(got[offs[b]:offs[b] + n] - want)
        assert err.max() < 2e-2 and err.mean() < 2e-3, (b, err.max(), err.mean())
    assert bi.bi_device_status() == 0


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 8, 64), (16, 4, 128)])
def test_fp8_cache_decode_rows_equal_prefill_rows(Hq, Hkv, hd):
    """Prefill of whole sequences, chunked prefill and single-token decode steps all
    write the same FP8 history and read it through the same gather + attention."""
    rng = np.random.default_rng(7 + hd)
    lens = [600, 65, 1030]
    T = sum(lens)
    kb, vb = normal_bf16(rng, (T, Hkv, hd), 1.0), normal_bf16(rng, (T, Hkv, hd), 1.0)
    qb = normal_bf16(rng, (T, Hq, hd), 1.0)
    offs = np.concatenate([[0], np.cumsum(lens)])
    full_c = Fp8Cache(lens, Hkv, hd, np.random.default_rng(1))
    full_c.write([(b, 0, n) for b, n in enumerate(lens)], kb, vb)
    full, *_ = full_c.attend([(b, 0, n) for b, n in enumerate(lens)], qb, Hq, max(lens))
    # another cache written in chunks of 97, read back one decode row at a few positions
    chunked = Fp8Cache(lens, Hkv, hd, np.random.default_rng(2))
    for b, n in enumerate(lens):
        for s0 in range(0, n, 97):
            e = min(n, s0 + 97)
            rows = slice(offs[b] + s0, offs[b] + e)
            chunked.write([(b, s0, e - s0)], kb[rows], vb[rows])
    for pos in (0, 64, 511, 599, 1029):
        pcs = [(b, pos, 1) for b, n in enumerate(lens) if pos < n]
        rows = [offs[b] + pos for b, n in enumerate(lens) if pos < n]
        for max_ctx in (2048, 8192):
            o, *_ = chunked.attend(pcs, qb[rows], Hq, max_ctx)
            assert same_bits(o, full[torch.tensor(rows, device="cuda")]), (pos, max_ctx)


@pytest.mark.parametrize("Hq,Hkv,hd", [(8, 8, 64), (16, 4, 128), (8, 1, 128)])
def test_direct_fp8_attention_equals_gather_path(Hq, Hkv, hd):
    """Reading the FP8 pages inside attention gives the bits of gather + bf16
    attention: whole-sequence prefill, prefill chunks that start mid-sequence
    (slots after them hold NaN codes and scales) and decode rows; the fused
    output quantisation equals bi_quantize_fp8 of the bf16 output."""
    rng = np.random.default_rng(11 + hd + Hkv)
    lens = [300, 1, 129, 700, 64]
    T = sum(lens)
    kb, vb = normal_bf16(rng, (T, Hkv, hd), 1.0), normal_bf16(rng, (T, Hkv, hd), 1.0)
    qb = normal_bf16(rng, (T, Hq, hd), 1.0)
    offs = np.concatenate([[0], np.cumsum(lens)])
    c = Fp8Cache(lens, Hkv, hd, rng)
    # only the first part of each sequence is in the cache: the rest stays NaN
    part = [max(1, n // 2) for n in lens]
    c.write([(b, 0, n) for b, n in enumerate(part)], np.concatenate([kb[offs[b]:offs[b] + n] for b, n in enumerate(part)]),
            np.concatenate([vb[offs[b]:offs[b] + n] for b, n in enumerate(part)]))
    cases = {
        "prefill": [(b, 0, n) for b, n in enumerate(part)],
        "chunk": [(b, max(0, n - 37), min(37, n)) for b, n in enumerate(part)],
        "decode": [(b, n - 1, 1) for b, n in enumerate(part)],
    }
    for name, pcs in cases.items():
        rows = np.concatenate([offs[b] + np.arange(p0, p0 + n) for b, p0, n in pcs])
        for max_ctx in (max(part), 4096):
            ref, *_ = c.attend(pcs, qb[rows], Hq, max_ctx)
            got, oq, osc = c.attend_direct(pcs, qb[rows], Hq, max_ctx, quant=True)
            assert same_bits(got, ref), (name, max_ctx)
            wq = torch.empty_like(oq)
            ws_ = torch.empty_like(osc)
            bi.bi_quantize_fp8(ref, ref.shape[0], ref.shape[1], 1, wq, ws_)
            assert torch.equal(oq, wq) and same_bits(osc, ws_), (name, max_ctx)
            assert not torch.isnan(got.float()).any()
    assert bi.bi_device_status() == 0


@pytest.mark.parametrize("hd,lo,hi", [(64, -12, 1), (128, -12, 1), (64, -30, 5), (128, -30, 5)])
def test_direct_fp8_attention_every_code(hd, lo, hi):
    """Every finite e4m3 code (zeros and subnormals included) under scales 2^lo ..
    2^(hi-1), read directly by attention (per-CTA and persistent decode
    schedules, prefill), against the gather path: the same bits wherever the
    output is above 2^-100.  Below that, in outputs within a few ulps of fp32's
    smallest normal number, P.V terms under 2^-126 (fp32 subnormals, which the
    two paths form from differently scaled operands) may round differently; the
    difference stays under 2^-124.  (Every phase reads through the direct path,
    so decode, prefill and recompute still agree bit for bit.)"""
    Hq, Hkv = 8, 2
    rng = np.random.default_rng(hd)
    lens = [2500, 700]
    c = Fp8Cache(lens, Hkv, hd, rng)
    codes = np.concatenate([np.arange(0x00, 0x7F), np.arange(0x80, 0xFF)]).astype(np.uint8)   # 254 finite codes
    for t in (c.k8, c.v8):
        fill = codes[rng.integers(0, len(codes), t.numel())]
        fill[: len(codes)] = codes                       # every code at least once
        t.copy_(torch.from_numpy(fill.reshape(t.shape)))
    for t in (c.ks, c.vs):
        t.copy_(torch.from_numpy((2.0 ** rng.integers(lo, hi, t.shape)).astype(np.float32)))
    qb = normal_bf16(rng, (sum(lens), Hq, hd), 1.0)
    offs = np.concatenate([[0], np.cumsum(lens)])
    for pcs in ([(0, 0, lens[0]), (1, 0, lens[1])], [(0, lens[0] - 1, 1), (1, lens[1] - 1, 1)],
                [(0, 1000, 200), (1, 500, 200)]):
        rows = np.concatenate([offs[b] + np.arange(p0, p0 + n) for b, p0, n in pcs])
        for max_ctx in (2560, 8192):
            ref, *_ = c.attend(pcs, qb[rows], Hq, max_ctx)
            got, *_ = c.attend_direct(pcs, qb[rows], Hq, max_ctx)
            r, g = host_f32(ref), host_f32(got)
            d = np.abs(r - g)
            big = np.abs(r) >= 2.0 ** -100
            assert np.array_equal(r[big].view(np.uint32), g[big].view(np.uint32)), (pcs[0], max_ctx)
            assert d.max() <= 2.0 ** -124, (pcs[0], max_ctx, d.max())
    assert bi.bi_device_status() == 0
