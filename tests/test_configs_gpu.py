"""Full-size workloads: bitwise invariance across batch compositions and oracle parity.

  * logprob head: 8 sequences x 64 tokens, d 256, V 4096 (RMSNorm + lm_head + log-softmax + gather)
  * MoE FFN layer: 4096 tokens, 64 experts, top-8, d 2048, F 1024
  * large-vocab logprob: 16384 rows, d 4096, V 129280 (lm_head + fp32 log-softmax + gather)
  * long-context GQA decoder: 8 layers, d 2048, 16/4 heads x 128, ragged contexts 1K-32K
"""
import math

import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from invariant_forward_policy_gb300.decoder import Decoder
from oracle import model as omodel
from oracle import moe as omoe
from oracle import ops
from synthetic import (C1, C3, C4, C5, bits_to_f32, make_c5_prompt_lengths, make_decoder_weights, make_logprob_head,
                       make_moe_layer)
from tests.gpu_util import dev_bf16, same_bits
from tests.parity import E2E_MAX_LONG, E2E_MEAN_LONG, anchored_parity, e2e_close

pytestmark = pytest.mark.gpu


def _head(h, g, W, ids, norm=True):
    """RMSNorm (optional) -> fp32 lm_head GEMM -> logprob of ids, all through the C ABI."""
    T, d = h.shape
    V = W.shape[0]
    x = torch.empty_like(h)
    if norm:
        bi.bi_rmsnorm(h, None, g, x, T, d, 1e-6)
    else:
        x = h
    logits = torch.empty((T, V), dtype=torch.float32, device="cuda")
    bi.bi_gemm(x, T, d, W, V, logits, bi.BI_DTYPE_FP32)
    lp = torch.empty(T, dtype=torch.float32, device="cuda")
    bi.bi_logprob_gather(logits, ids, T, V, lp)
    return lp


# ----------------------------------------------------------------------------- logprob head
def test_logprob_head_invariant_over_batch_sizes_and_orders():
    c = C1
    n = c["n_seq"] * c["seq_len"]
    inp = make_logprob_head(n, c["d"], c["vocab"], c["w_std"], c["seed"])
    h, g, W = dev_bf16(inp["h"]), dev_bf16(inp["gain"]), dev_bf16(inp["w"])
    ids = torch.from_numpy(inp["ids"]).cuda()
    full = _head(h, g, W, ids)
    _, want = omodel.logprob_head(bits_to_f32(inp["h"]), bits_to_f32(inp["gain"]), bits_to_f32(inp["w"]), inp["ids"])
    err = np.abs(full.cpu().numpy() - want)
    assert err.max() < 1e-4, err.max()
    seqs = np.random.default_rng(c["seed"]).permutation(c["n_seq"])
    L = c["seq_len"]
    for bs in range(1, c["n_seq"] + 1):                       # batch sizes 1..8
        rows = np.concatenate([np.arange(s * L, (s + 1) * L) for s in seqs[:bs]])
        r = torch.from_numpy(rows).cuda()
        assert same_bits(_head(h[r].contiguous(), g, W, ids[r].contiguous()), full[r]), bs
    for k in range(5):                                          # shuffled orders
        rows = np.random.default_rng(100 + k).permutation(n)
        r = torch.from_numpy(rows).cuda()
        assert same_bits(_head(h[r].contiguous(), g, W, ids[r].contiguous()), full[r]), k


# ----------------------------------------------------------------------------- MoE layer
def _moe(x, lg, w13, w2, c, mode=bi.BI_INVARIANT):
    T = x.shape[0]
    out = torch.empty((T, c["d"]), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bi.bi_moe_layer_workspace_size(T, c["d"], c["n_experts"], c["top_k"], c["ffn"], mode),
                     dtype=torch.uint8, device="cuda")
    bi.bi_moe_layer(x, lg, T, c["d"], c["n_experts"], c["top_k"], c["ffn"], w13, w2, out, mode, ws)
    return out


def test_moe_layer_full_size_invariance_and_oracle():
    c = C3
    inp = make_moe_layer(c["n_tokens"], c["d"], c["ffn"], c["n_experts"], c["w_std"], c["seed"])
    x, lg = dev_bf16(inp["x"]), torch.from_numpy(inp["router_logits"]).cuda()
    w13, w2 = dev_bf16(inp["w13"]), dev_bf16(inp["w2"])
    T = c["n_tokens"]
    full = _moe(x, lg, w13, w2, c)
    # 16 batches of 256
    parts = [_moe(x[i:i + 256].contiguous(), lg[i:i + 256].contiguous(), w13, w2, c) for i in range(0, T, 256)]
    assert same_bits(torch.cat(parts), full)
    # random sizes from {1..1024} over a shuffled token order
    rng = np.random.default_rng(c["seed"])
    perm = rng.permutation(T)
    i = 0
    while i < T:
        n = int(rng.integers(1, 1025))
        r = torch.from_numpy(perm[i:i + n]).cuda()
        assert same_bits(_moe(x[r].contiguous(), lg[r].contiguous(), w13, w2, c), full[r])
        i += n
    # oracle on 256 tokens
    sub = np.sort(rng.choice(T, 256, replace=False))
    want, _, _ = omoe.moe_layer(bits_to_f32(inp["x"][sub]), inp["router_logits"][sub], bits_to_f32(inp["w13"]),
                                bits_to_f32(inp["w2"]), c["top_k"])
    got = full[torch.from_numpy(sub).cuda()].float().cpu().numpy()
    err = np.abs(got - want)
    # two bf16 roundings (expert output, combine) plus dot-product order inside the experts
    assert np.all(err <= 2 * 2.0 ** -7 * np.abs(want) + 2e-2), err.max()
    assert np.mean(err) < 2e-3
    # the non-invariant path computes the same layer approximately
    fast = _moe(x, lg, w13, w2, c, bi.BI_FAST).float()
    assert torch.max(torch.abs(fast - full.float())).item() < 5e-2


# ----------------------------------------------------------------------------- large vocab
def test_large_vocab_logprob_two_partitions_k3_zero():
    c = C4
    inp = make_logprob_head(c["n_tokens"], c["d"], c["vocab"], c["w_std"], c["seed"])
    h, W = dev_bf16(inp["h"]), dev_bf16(inp["w"])
    ids = torch.from_numpy(inp["ids"]).cuda()
    T = c["n_tokens"]
    lp_a = _head(h, None, W, ids, norm=False)                  # partition A: one batch
    rng = np.random.default_rng(c["seed"] + 1)
    perm = rng.permutation(T)
    lp_b = torch.empty_like(lp_a)
    i = 0
    while i < T:                                               # partition B: random sizes, shuffled
        n = int(rng.integers(1, 4097))
        r = torch.from_numpy(perm[i:i + n]).cuda()
        lp_b[r] = _head(h[r].contiguous(), None, W, ids[r].contiguous(), norm=False)
        i += n
    s = ops.diff_stats(lp_a.cpu().numpy(), lp_b.cpu().numpy())
    assert s == {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}, s
    sub = np.sort(rng.choice(T, 48, replace=False))
    _, want = omodel.logprob_head(bits_to_f32(inp["h"][sub]), None, bits_to_f32(inp["w"]), inp["ids"][sub],
                                  norm=False)
    err = np.abs(lp_a.cpu().numpy()[sub] - want)
    assert err.max() < 2e-4, err.max()
    # the fused lm_head + log-softmax (no logits in memory): same two partitions
    d = c["d"]

    def fused(hh, ii):
        n = hh.shape[0]
        out = torch.empty(n, dtype=torch.float32, device="cuda")
        ws = torch.empty(bi.bi_lm_head_logprob_workspace_size(n, c["vocab"], d), dtype=torch.uint8, device="cuda")
        bi.bi_lm_head_logprob(hh, n, d, W, c["vocab"], ii, out, None, bi.BI_INVARIANT, ws)
        return out

    fa = fused(h, ids)
    fb = torch.empty_like(fa)
    rng = np.random.default_rng(c["seed"] + 2)
    perm = rng.permutation(T)
    i = 0
    while i < T:
        n = int(rng.integers(1, 4097))
        r = torch.from_numpy(perm[i:i + n]).cuda()
        fb[r] = fused(h[r].contiguous(), ids[r].contiguous())
        i += n
    s = ops.diff_stats(fa.cpu().numpy(), fb.cpu().numpy())
    assert s == {"max": 0.0, "mean": 0.0, "std": 0.0, "k3": 0.0}, s
    errf = np.abs(fa.cpu().numpy()[sub] - want)
    assert errf.max() < 2e-4, errf.max()


# ----------------------------------------------------------------------------- long-context GQA
@pytest.mark.slow
def test_long_context_gqa_decoder_diff_zero():
    """64 ragged sequences (contexts 1K-32K, log-uniform), page 64, split 512,
    chunk 2048.  Rollout of 64 greedy tokens as one decode batch of 64 and as
    subsets of 1, 7 and 33 sequences in shuffled order; prefill chunks 2048 and
    1536; recompute with chunk 2048 and with 4096 in another packing order.
    Every logprob is bit-equal; the oracle agrees on the two shortest sequences
    and on the one whose prompt is nearest 4096 tokens."""
    c = C5
    shape = c["shape"]
    n_gen = 64
    wb = make_decoder_weights(shape, seed=c["seed"], w_std=c["w_std"])
    lens = make_c5_prompt_lengths(c["batch"], c["ctx_min"], c["ctx_max"], c["seed"])
    rng = np.random.default_rng(c["seed"] + 3)
    prompts = [rng.integers(0, shape.vocab, int(n)).astype(np.int32) for n in lens]
    max_pos = int(lens.max()) + n_gen + 64
    dec = Decoder(shape, wb, max_pos=max_pos)
    B = len(prompts)
    mb = -(-(int(lens.max()) + n_gen) // 64)

    def rollout(idx, chunk, seed):
        bt, nb = dec.paged_block_table([len(prompts[i]) + n_gen for i in idx], mb, seed=seed)
        cache = dec.alloc_cache(nb)
        return dec.rollout([prompts[i] for i in idx], n_gen, cache, bt, chunk=chunk, prefill_max_tokens=16384)

    ids, lp = rollout(list(range(B)), c["chunk"], 1)
    torch.cuda.synchronize()
    order = rng.permutation(B)
    o = 0
    for n_sub, chunk in ((1, 1536), (7, 2048), (33, 2048)):
        idx = [int(i) for i in order[o:o + n_sub]]
        o += n_sub
        i2, l2 = rollout(idx, chunk, 10 + n_sub)
        t = torch.tensor(idx, device="cuda")
        assert torch.equal(i2, ids[t]) and same_bits(l2, lp[t]), n_sub
        del i2, l2
        torch.cuda.empty_cache()
    gens = ids.cpu().numpy()
    for chunk, pack in ((2048, None), (4096, [int(i) for i in order])):
        bt, nb = dec.paged_block_table([len(p) + n_gen for p in prompts], mb, seed=7)
        cache = dec.alloc_cache(nb)
        lt = dec.recompute(prompts, gens, cache, bt, chunk=chunk, order=pack, max_tokens=16384)
        assert same_bits(lt, lp), chunk
        del cache
        torch.cuda.empty_cache()
    W = omodel.weights_to_f32(wb)
    errs = []
    short = np.argsort(lens)[:2]
    near_4k = int(np.argmin(np.abs(lens - 4096)))           # 9 splits deep, scored by the oracle too
    for b in list(short) + [near_4k]:
        _, want, _ = omodel.score_generation(W, shape, prompts[b], gens[b])
        errs.append(e2e_close(lp[b].cpu().numpy(), want, E2E_MAX_LONG, E2E_MEAN_LONG))
        print("  sequence %d (prompt %d): max %.2e mean %.2e" % (b, lens[b], errs[-1].max(), errs[-1].mean()))
    errs = np.concatenate(errs)
    print("GQA long-context free-running oracle error: max %.2e mean %.2e" % (errs.max(), errs.mean()))
    anchored_parity(dec, wb, shape, [np.concatenate([prompts[short[0]], gens[short[0]][:-1]])], seed=5)
    assert bi.bi_device_status() == 0
