"""Block-FP8 decoder ("vLLM Achieves Bitwise-Consistent RL Training ..." §4.1 W8A8
linear layers, §4.2 FP8 KV cache) end to end: rollout (prefill + decode, graph
and eager, staggered batches) and the training recompute (any chunking and
packing) give the same bits; the FP8 cache holds the oracle's codes; every layer
agrees with the FP8 oracle from the GPU's own input, within the FP8 bounds."""
import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from invariant_forward_policy_gb300.decoder import Decoder
from oracle import fp8 as ofp8
from oracle import model as omodel
from oracle import ops
from synthetic import DecoderShape, make_decoder_weights, make_prompts
from tests.gpu_util import same_bits
from tests.parity import E2E_MAX_FP8, E2E_MEAN_FP8, anchored_parity, e2e_close
from tests.test_decoder_gpu import staggered_rollout

pytestmark = pytest.mark.gpu


def _fp8_decoder(shape, seed, max_pos, w_std=0.05):
    wb = make_decoder_weights(shape, seed=seed, w_std=w_std)
    return Decoder(shape, wb, max_pos=max_pos, fp8=True), wb


def _cache_layer(dec, cache, layer, which):
    """(codes [n_blocks, Hkv, 64, hd] uint8, scales [n_blocks, Hkv, 64] fp32) of one layer's K or V."""
    s = dec.shape
    nb = cache.n_blocks
    n_codes = nb * s.n_heads_kv * 64 * s.head_dim
    buf = (cache.k if which == "k" else cache.v)[layer]
    codes = buf[:n_codes].view(nb, s.n_heads_kv, 64, s.head_dim).cpu().numpy()
    scales = buf[n_codes:n_codes + nb * s.n_heads_kv * 64 * 4].view(torch.float32).view(nb, s.n_heads_kv, 64)
    return codes, scales.cpu().numpy()


def test_fp8_decoder_rollout_equals_recompute_and_oracle():
    shape = DecoderShape(2, 256, 4, 2, 64, 512, 1024)
    dec, wb = _fp8_decoder(shape, seed=51, max_pos=1024)
    prompts = make_prompts(5, 10, 150, shape.vocab, seed=52)
    n_gen = 40
    max_ctx = max(len(p) for p in prompts) + n_gen
    mb = -(-max_ctx // 64)
    cache = dec.alloc_cache(5 * mb + 3)
    bt = dec.block_table(5, mb, seed=4)
    ids_g, lp_g = dec.rollout(prompts, n_gen, cache, bt, use_graph=True)
    cache_e = dec.alloc_cache(5 * mb + 3)
    ids_e, lp_e = dec.rollout(prompts, n_gen, cache_e, bt, use_graph=False)
    assert torch.equal(ids_g, ids_e) and same_bits(lp_g, lp_e)          # graph == eager
    assert torch.equal(cache.k, cache_e.k) and torch.equal(cache.v, cache_e.v)
    gens = ids_g.cpu().numpy()
    for chunk, order in ((2048, None), (64, [4, 2, 0, 1, 3]), (97, [1, 0, 4, 3, 2])):
        c2 = dec.alloc_cache(5 * mb + 3)
        lp_t = dec.recompute(prompts, gens, c2, bt, chunk=chunk, order=order)
        s = ops.diff_stats(lp_g.cpu().numpy().ravel(), lp_t.cpu().numpy().ravel())
        assert s == {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}, (chunk, order, s)
        assert same_bits(lp_t, lp_g), (chunk, order)
    ids_s, lp_s = staggered_rollout(dec, prompts, n_gen, seed=5, max_ctx=max_ctx)
    assert torch.equal(ids_s, ids_g) and same_bits(lp_s, lp_g)
    anchored_parity(dec, wb, shape, [np.concatenate([prompts[b], gens[b][:-1]]) for b in range(5)], fp8=True)
    W8 = omodel.fp8_weights(omodel.weights_to_f32(wb))
    errs = []
    for b in range(5):
        _, want, _ = omodel.score_generation(W8, shape, prompts[b], gens[b])
        errs.append(e2e_close(lp_g[b].cpu().numpy(), want, E2E_MAX_FP8, E2E_MEAN_FP8))
    errs = np.concatenate(errs)
    print("FP8 free-running oracle error: max %.2e mean %.2e" % (errs.max(), errs.mean()))
    assert bi.bi_device_status() == 0


def test_fp8_cache_holds_the_oracle_codes():
    """Layer 0 reads the exact embedding, so its K and V codes and scales are the
    oracle's (RMSNorm, W8A8 QKV GEMM, RoPE, per-(token, head) quantisation) up to
    the rare e4m3 code that a differently summed GEMM output moves by one step."""
    shape = DecoderShape(2, 256, 8, 2, 128, 512, 1024)
    dec, wb = _fp8_decoder(shape, seed=61, max_pos=2048)
    prompts = make_prompts(3, 100, 700, shape.vocab, seed=62)
    mb = max(-(-len(p) // 64) for p in prompts)
    cache = dec.alloc_cache(3 * mb + 1)
    bt = dec.block_table(3, mb, seed=9)
    dec.prefill(prompts, cache, bt, chunk=256)
    W8 = omodel.fp8_weights(omodel.weights_to_f32(wb))
    lw = W8["layers"][0]
    hq, hkv, hd = shape.n_heads_q, shape.n_heads_kv, shape.head_dim
    kc, ks = _cache_layer(dec, cache, 0, "k")
    vc, vs = _cache_layer(dec, cache, 0, "v")
    tab = bt.cpu().numpy()
    n_code = n_code_eq = n_scale = n_scale_eq = 0
    for b, p in enumerate(prompts):
        n = len(p)
        x, _ = ops.rmsnorm(W8["embed"][np.asarray(p)], lw["attn_norm"], shape.eps)
        qkv = omodel.linear_fp8(x, *lw["fp8"]["wqkv"])
        k = ops.rope(qkv[:, hq * hd:(hq + hkv) * hd].reshape(n, hkv, hd), np.arange(n), shape.rope_theta)
        v = qkv[:, (hq + hkv) * hd:].reshape(n, hkv, hd)
        for got_c, got_s, t in ((kc, ks, k), (vc, vs, v)):
            wc, wsc = ofp8.quantize_blocks(t.reshape(n * hkv, hd), 1, block_cols=hd)
            gc = got_c[tab[b]].transpose(0, 2, 1, 3).reshape(-1, hkv, hd)[:n].reshape(n * hkv, hd)
            gs = got_s[tab[b]].transpose(0, 2, 1).reshape(-1, hkv)[:n].reshape(n * hkv)
            # where the vector's scale agrees, a moved code is one e4m3 step away
            # (adjacent magnitude, same sign) or a zero of the other sign
            diff = gc != wc
            same_scale = (gs == wsc[:, 0])[:, None]
            step = np.abs(gc.astype(np.int32) - wc.astype(np.int32)) <= 1
            zeros = ((gc & 0x7F) == 0) & ((wc & 0x7F) == 0)
            assert np.all(~diff | step | zeros | ~same_scale)
            n_code += gc.size
            n_code_eq += int((~diff).sum())
            n_scale += gs.size
            n_scale_eq += int((gs == wsc[:, 0]).sum())
    assert n_code_eq / n_code >= 0.995, n_code_eq / n_code
    assert n_scale_eq / n_scale >= 0.999, n_scale_eq / n_scale
    assert bi.bi_device_status() == 0


def test_fp8_gqa_long_context_rollout_equals_recompute():
    """GQA 8/2 with hd 128, contexts across several 512-position splits, in both
    modes: the invariant mode gives recompute == rollout bitwise; the fast mode
    runs the same layer with batch-shaped reductions and stays within the FP8
    oracle bounds."""
    shape = DecoderShape(2, 256, 8, 2, 128, 512, 1024)
    dec, wb = _fp8_decoder(shape, seed=71, max_pos=4096)
    prompts = make_prompts(4, 500, 1500, shape.vocab, seed=72)
    n_gen = 16
    max_ctx = max(len(p) for p in prompts) + n_gen
    mb = -(-max_ctx // 64)
    cache = dec.alloc_cache(4 * mb)
    bt = dec.block_table(4, mb, seed=6)
    ids, lp = dec.rollout(prompts, n_gen, cache, bt, chunk=512)
    gens = ids.cpu().numpy()
    c2 = dec.alloc_cache(4 * mb)
    lp_t = dec.recompute(prompts, gens, c2, bt, chunk=2048, order=[3, 1, 2, 0])
    assert same_bits(lp_t, lp)
    c3 = dec.alloc_cache(4 * mb)
    ids_f, lp_f = dec.rollout(prompts, n_gen, c3, bt, chunk=512, mode=bi.BI_FAST)
    W8 = omodel.fp8_weights(omodel.weights_to_f32(wb))
    for b in (0, 3):
        _, want, _ = omodel.score_generation(W8, shape, prompts[b], gens[b])
        e2e_close(lp[b].cpu().numpy(), want, E2E_MAX_FP8, E2E_MEAN_FP8)
    gf = ids_f.cpu().numpy()
    _, want_f, _ = omodel.score_generation(W8, shape, prompts[1], gf[1])
    e2e_close(lp_f[1].cpu().numpy(), want_f, E2E_MAX_FP8, E2E_MEAN_FP8)
    assert bi.bi_device_status() == 0
