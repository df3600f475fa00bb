"""Decoder handle: device weights, paged KV cache, rollout and training recompute.

The two halves of the article's RL loop ("vLLM Achieves Bitwise-Consistent RL
Training ...", §2 and §3.1) on one GPU:
  * rollout  — prefill the prompts, then greedy decode steps (optionally
               replayed from a CUDA graph, §4.6), each step emitting the sampled
               token and its logprob;
  * recompute — the training side scores the same tokens with one packed,
               chunked prefill over prompt + response.
Both call the same C entry points (bi_forward_prefill / bi_forward_decode),
which run the same kernels.  This module only allocates memory, fills
argument structures and sequences calls; no arithmetic of the forward runs here.
"""
from __future__ import annotations

import ctypes
import dataclasses

import numpy as np
import torch

from . import _lib as L


def _bf16_tensor(bits: np.ndarray, device) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
    return t.to(device)


# ------------------------------------------------------------ host bookkeeping
def block_ids(n_seq: int, max_blocks: int, seed: int | None = None, base: int = 0) -> np.ndarray:
    """Physical block ids [n_seq, max_blocks] (int32): base .. base + n_seq * max_blocks - 1,
    scattered over the cache by a seeded permutation (in order when seed is None)."""
    n = n_seq * max_blocks
    ids = np.arange(n, dtype=np.int32) + base
    if seed is not None:
        ids = np.random.default_rng(seed).permutation(ids).astype(np.int32)
    return ids.reshape(n_seq, max_blocks)


def paged_block_ids(ctx_lens, max_blocks: int, seed: int | None = None):
    """Block table giving sequence b only ceil(ctx_lens[b] / 64) physical blocks
    (entries past that are -1), scattered over the cache by a seeded permutation.
    Returns (table [n_seq, max_blocks] int32, n_blocks)."""
    need = [-(-int(n) // 64) for n in ctx_lens]
    total = int(sum(need))
    ids = np.arange(total, dtype=np.int32)
    if seed is not None:
        ids = np.random.default_rng(seed).permutation(ids).astype(np.int32)
    tab = np.full((len(need), max_blocks), -1, dtype=np.int32)
    o = 0
    for b, n in enumerate(need):
        tab[b, :n] = ids[o:o + n]
        o += n
    return tab, total


def recompute_pack(prompts, gens, order):
    """The training side's packed batch, sequence by sequence in `order`: tokens
    [prompt, gen[:-1]], targets (gen from row len(prompt) - 1 on, 0 before) and the
    first scored row len(prompt) - 1."""
    seqs, tg, lf = [], [], []
    for b in order:
        p = np.asarray(prompts[b], np.int32)
        g = np.asarray(gens[b], np.int32)
        s = np.concatenate([p, g[:-1]])
        t = np.zeros(len(s), np.int32)
        t[len(p) - 1:] = g
        seqs.append(s)
        tg.append(t)
        lf.append(len(p) - 1)
    return seqs, tg, lf


def recompute_rows(prompt_lens, n_gen: int):
    """Rows of the same packed batch on static buffers, sequences in order: cu
    (B + 1 offsets), p_dst (the prompts' rows, concatenated), g_dst [B, n_gen - 1]
    (the rows of the fed-back generated tokens; None when n_gen == 1) and t_dst
    [B, n_gen] (the rows whose target is generated token k)."""
    lens = np.asarray(prompt_lens, dtype=np.int64)
    cu = np.concatenate([[0], np.cumsum(lens + n_gen - 1)])
    pd, gd, td = [], [], []
    for b in range(len(lens)):
        o = cu[b]
        pd.append(o + np.arange(lens[b]))
        gd.append(o + lens[b] + np.arange(n_gen - 1))
        td.append(o + lens[b] - 1 + np.arange(n_gen))
    return cu, np.concatenate(pd), (np.stack(gd) if n_gen > 1 else None), np.stack(td)


@dataclasses.dataclass
class KVCache:
    k: torch.Tensor
    v: torch.Tensor
    n_blocks: int


class Decoder:
    """A decoder whose weights live in caller-owned (torch) device memory."""

    def __init__(self, shape, weight_bits: dict, max_pos: int, device="cuda", fp8: bool = False):
        """fp8: block-FP8 W8A8 linear layers and an FP8 KV cache.  The FP8 copies
        of the four linear weights of every layer are made here from the bf16
        masters by the deployment rule (bi_quantize_fp8, 128 x 128 blocks) and
        kept; a trainer that updates the masters re-runs `requantize()`."""
        self.shape = shape
        self.device = torch.device(device)
        self.fp8 = bool(fp8)
        s = shape
        self.cfg = L.bi_model_config(n_layers=s.n_layers, d=s.d, n_heads_q=s.n_heads_q, n_heads_kv=s.n_heads_kv,
                                     head_dim=s.head_dim, ffn=s.ffn, vocab=s.vocab, eps=s.eps,
                                     rope_theta=s.rope_theta, kv_block=64, kv_split=s.kv_split, max_pos=max_pos,
                                     fp8=1 if fp8 else 0)
        dev = self.device
        self.w = {k: _bf16_tensor(weight_bits[k], dev) for k in ("embed", "final_norm", "lm_head")}
        self.layers = [{k: _bf16_tensor(v, dev) for k, v in lw.items()} for lw in weight_bits["layers"]]
        self.rope_table = torch.empty((max_pos, s.head_dim), dtype=torch.float32, device=dev)
        if self.fp8:
            for lw in self.layers:
                for k in ("wqkv", "wo", "w13", "w2"):
                    N, K = lw[k].shape
                    lw[k + "8"] = torch.empty((N, K), dtype=torch.uint8, device=dev)
                    lw[k + "_s"] = torch.empty((-(-N // 128), K // 128), dtype=torch.float32, device=dev)
            self.requantize()

        def ptr(lw, k):
            return lw[k].data_ptr() if k in lw else None

        lw_arr = (L.bi_layer_weights * s.n_layers)()
        for i, lw in enumerate(self.layers):
            lw_arr[i] = L.bi_layer_weights(lw["attn_norm"].data_ptr(), lw["wqkv"].data_ptr(), lw["wo"].data_ptr(),
                                           lw["ffn_norm"].data_ptr(), lw["w13"].data_ptr(), lw["w2"].data_ptr(),
                                           ptr(lw, "wqkv8"), ptr(lw, "wqkv_s"), ptr(lw, "wo8"), ptr(lw, "wo_s"),
                                           ptr(lw, "w138"), ptr(lw, "w13_s"), ptr(lw, "w28"), ptr(lw, "w2_s"))
        self._lw_arr = lw_arr
        self._weights = L.bi_weights(self.w["embed"].data_ptr(), self.w["final_norm"].data_ptr(),
                                     self.w["lm_head"].data_ptr(), ctypes.cast(lw_arr, ctypes.POINTER(L.bi_layer_weights)),
                                     self.rope_table.data_ptr())
        self.handle = L.bi_model_create(self.cfg, self._weights)
        self.max_pos = max_pos

    def requantize(self):
        """FP8 copies of the linear weights from the bf16 masters (128 x 128 blocks)."""
        for lw in self.layers:
            for k in ("wqkv", "wo", "w13", "w2"):
                N, K = lw[k].shape
                L.bi_quantize_fp8(lw[k], N, K, 128, lw[k + "8"], lw[k + "_s"])

    def close(self):
        if getattr(self, "handle", None):
            L.bi_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # ------------------------------------------------------------ memory
    def alloc_cache(self, n_blocks: int) -> KVCache:
        s = self.shape
        if self.fp8:
            # per layer: e4m3 codes [n_blocks, Hkv, 64, hd], then fp32 scales [n_blocks, Hkv, 64]
            per_layer = L.bi_kv_cache_bytes(self.cfg, n_blocks) // s.n_layers
            return KVCache(torch.zeros((s.n_layers, per_layer), dtype=torch.uint8, device=self.device),
                           torch.zeros((s.n_layers, per_layer), dtype=torch.uint8, device=self.device), n_blocks)
        shape = (s.n_layers, n_blocks, s.n_heads_kv, 64, s.head_dim)
        return KVCache(torch.zeros(shape, dtype=torch.bfloat16, device=self.device),
                       torch.zeros(shape, dtype=torch.bfloat16, device=self.device), n_blocks)

    def block_table(self, n_seq: int, max_blocks: int, seed: int | None = None, base: int = 0) -> torch.Tensor:
        """Physical blocks for n_seq sequences; a seeded permutation scatters them over the cache."""
        return torch.from_numpy(block_ids(n_seq, max_blocks, seed, base)).to(self.device)

    def paged_block_table(self, ctx_lens, max_blocks: int, seed: int | None = None):
        """Block table giving sequence b only ceil(ctx_lens[b] / 64) physical blocks
        (entries past that are -1 and never touched), scattered over the cache by a
        seeded permutation.  Returns (table [n_seq, max_blocks] int32, n_blocks)."""
        tab, total = paged_block_ids(ctx_lens, max_blocks, seed)
        return torch.from_numpy(tab).to(self.device), total

    def workspace(self, max_tokens, max_pieces, max_ctx, max_logit_rows, mode=L.BI_INVARIANT) -> torch.Tensor:
        n = L.bi_forward_workspace_size(self.cfg, max_tokens, max_pieces, max_ctx, max_logit_rows, mode)
        return torch.empty(n, dtype=torch.uint8, device=self.device)

    # ------------------------------------------------------------ calls
    def prefill(self, seqs, cache: KVCache, block_table: torch.Tensor, start_pos=None, logit_from=None,
                targets=None, chunk=2048, max_tokens=8192, max_ctx=None, max_logit_rows=2048,
                mode=L.BI_INVARIANT, workspace=None, tokens_dev=None, dump=None):
        """Packed prefill of a list of token arrays; returns (logprob [T], sampled [T]) over the packed rows.

        `dump` (bf16 [n_layers + 2, rows, d]) receives the per-layer residual
        stream of a single-pass call (see bi_model_set_dump)."""
        lens = [len(x) for x in seqs]
        B = len(seqs)
        cu = np.zeros(B + 1, dtype=np.int64)
        cu[1:] = np.cumsum(lens)
        T = int(cu[-1])
        start_pos = [0] * B if start_pos is None else list(start_pos)
        if max_ctx is None:
            max_ctx = max(int(sp) + n for sp, n in zip(start_pos, lens))
        if tokens_dev is None:
            tokens_dev = torch.from_numpy(np.concatenate([np.asarray(x, np.int32) for x in seqs])).to(self.device)
        tgt = None
        if targets is not None:
            tgt = torch.from_numpy(np.concatenate([np.asarray(x, np.int32) for x in targets])).to(self.device)
        lp = torch.full((T,), float("nan"), dtype=torch.float32, device=self.device)
        sm = torch.full((T,), -1, dtype=torch.int32, device=self.device)
        if workspace is None:
            workspace = self.workspace(max_tokens, min(B, 128), max_ctx, max_logit_rows, mode)
        if dump is not None:
            L.bi_model_set_dump(self.handle, dump, dump.shape[1])
        try:
            L.bi_forward_prefill(self.handle, tokens_dev, tgt, cu, start_pos, logit_from, B, chunk, block_table,
                                 block_table.shape[1], cache.k, cache.v, cache.n_blocks, lp, sm, workspace, max_tokens,
                                 max_ctx, max_logit_rows, mode)
        finally:
            if dump is not None:
                L.bi_model_set_dump(self.handle, None, 0)
        return lp, sm, cu

    def decode(self, tokens: torch.Tensor, pos: torch.Tensor, cache: KVCache, block_table: torch.Tensor, max_ctx: int,
               sampled: torch.Tensor, logprob: torch.Tensor, workspace: torch.Tensor, mode=L.BI_INVARIANT):
        L.bi_forward_decode(self.handle, tokens, pos, tokens.numel(), block_table, block_table.shape[1], cache.k,
                            cache.v, cache.n_blocks, max_ctx, sampled, logprob, workspace, mode)

    # ------------------------------------------------------------ RL halves
    def rollout(self, prompts, n_gen: int, cache: KVCache, block_table: torch.Tensor, chunk=2048, use_graph=True,
                mode=L.BI_INVARIANT, prefill_max_tokens=8192):
        """Greedy rollout: prefill, then n_gen - 1 decode steps.  Returns (ids [B, n_gen], lp [B, n_gen]) on device."""
        B = len(prompts)
        lens = np.array([len(p) for p in prompts])
        max_ctx = int(lens.max()) + n_gen
        dev = self.device
        lp0, sm0, cu = self.prefill(prompts, cache, block_table, logit_from=[n - 1 for n in lens], chunk=chunk,
                                    max_tokens=prefill_max_tokens, max_ctx=max_ctx, mode=mode)
        last = torch.from_numpy(cu[1:] - 1).to(dev)
        hist_ids = torch.zeros((n_gen, B), dtype=torch.int32, device=dev)
        hist_lp = torch.zeros((n_gen, B), dtype=torch.float32, device=dev)
        hist_ids[0] = sm0[last]
        hist_lp[0] = lp0[last]
        tok = hist_ids[0].clone()
        pos = torch.from_numpy(lens.astype(np.int32)).to(dev)
        step = torch.ones(1, dtype=torch.int32, device=dev)
        sampled = torch.zeros(B, dtype=torch.int32, device=dev)
        lp = torch.zeros(B, dtype=torch.float32, device=dev)
        ws = self.workspace(B, B, max_ctx, B, mode)

        def one_step():
            self.decode(tok, pos, cache, block_table, max_ctx, sampled, lp, ws, mode)
            L.bi_decode_advance(sampled, lp, tok, pos, B, step, hist_ids, hist_lp, n_gen)

        n_steps = n_gen - 1
        if n_steps <= 0:
            return hist_ids.T.contiguous(), hist_lp.T.contiguous()
        one_step()  # eager first step (also configures kernel attributes before any capture)
        if use_graph and n_steps > 1:
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                one_step()
            for _ in range(n_steps - 1):
                g.replay()
        else:
            for _ in range(n_steps - 1):
                one_step()
        return hist_ids.T.contiguous(), hist_lp.T.contiguous()

    def recompute(self, prompts, gens, cache: KVCache, block_table: torch.Tensor, chunk=2048, order=None,
                  mode=L.BI_INVARIANT, max_tokens=8192, max_logit_rows=2048):
        """Training-side scoring of prompt + response; returns lp [B, n_gen] (device).

        `order` packs the sequences in another order (a different batch layout)."""
        B = len(prompts)
        order = list(range(B)) if order is None else list(order)
        gens = [np.asarray(g, np.int32) for g in gens]
        seqs, tg, lf = recompute_pack(prompts, gens, order)
        bt = block_table[torch.as_tensor(order, device=block_table.device)]
        lp, _, cu = self.prefill(seqs, cache, bt, logit_from=lf, targets=tg, chunk=chunk, max_tokens=max_tokens,
                                 max_logit_rows=max_logit_rows, mode=mode)
        out = torch.empty((B, len(gens[0])), dtype=torch.float32, device=self.device)
        for j, b in enumerate(order):
            out[b] = lp[int(cu[j]) + lf[j]: int(cu[j + 1])]
        return out


class Episode:
    """One RL data step on static buffers: rollout of a fixed set of prompts
    (prefill + n_gen - 1 greedy decode steps replayed from one CUDA graph),
    then the training-side recompute of every sampled token's logprob with a
    single packed, chunked prefill.  All buffers and the decode graph are made
    once; `run()` only launches work (plus a few index copies that build the
    recompute's packed token array from the rollout's output)."""

    def __init__(self, dec: Decoder, prompt_lens, n_gen: int, chunk: int = 2048, mode=L.BI_INVARIANT,
                 max_tokens: int = 16384, max_logit_rows: int = 4096, block_seed: int = 1):
        self.dec, self.n_gen, self.chunk, self.mode = dec, n_gen, chunk, mode
        dev = dec.device
        lens = np.asarray(prompt_lens, dtype=np.int64)
        self.lens, B = lens, len(lens)
        self.B = B
        self.max_ctx = int(lens.max()) + n_gen
        mb = -(-self.max_ctx // 64)
        self.cache = dec.alloc_cache(B * mb)
        self.bt = dec.block_table(B, mb, seed=block_seed)
        self.max_tokens, self.max_logit_rows = max_tokens, max_logit_rows
        # prefill of the prompts
        self.cu_p = np.concatenate([[0], np.cumsum(lens)])
        self.T_p = int(self.cu_p[-1])
        self.lp_p = torch.zeros(self.T_p, dtype=torch.float32, device=dev)
        self.sm_p = torch.zeros(self.T_p, dtype=torch.int32, device=dev)
        self.last = torch.from_numpy(self.cu_p[1:] - 1).to(dev)
        # decode state
        self.tok = torch.zeros(B, dtype=torch.int32, device=dev)
        self.pos0 = torch.from_numpy(lens.astype(np.int32)).to(dev)
        self.pos = self.pos0.clone()
        self.step = torch.ones(1, dtype=torch.int32, device=dev)
        self.sampled = torch.zeros(B, dtype=torch.int32, device=dev)
        self.lp = torch.zeros(B, dtype=torch.float32, device=dev)
        self.hist_ids = torch.zeros((n_gen, B), dtype=torch.int32, device=dev)
        self.hist_lp = torch.zeros((n_gen, B), dtype=torch.float32, device=dev)
        # recompute: packed [prompt_b, gen_b[:-1]] per sequence
        self.cu_r, pd, gd, td = recompute_rows(lens, n_gen)
        self.T_r = int(self.cu_r[-1])
        self.p_dst = torch.from_numpy(pd).to(dev)
        self.g_dst = torch.from_numpy(gd).to(dev) if gd is not None else None
        self.t_dst = torch.from_numpy(td).to(dev)
        self.rec_tok = torch.zeros(self.T_r, dtype=torch.int32, device=dev)
        self.rec_tgt = torch.zeros(self.T_r, dtype=torch.int32, device=dev)
        self.rec_lp = torch.zeros(self.T_r, dtype=torch.float32, device=dev)
        self.cache_r = dec.alloc_cache(B * mb)
        self.ws_p = dec.workspace(max_tokens, min(B, 128), self.max_ctx, max_logit_rows, mode)
        self.ws_d = dec.workspace(B, B, self.max_ctx, B, mode)
        self.graph = None

    def _decode_step(self):
        self.dec.decode(self.tok, self.pos, self.cache, self.bt, self.max_ctx, self.sampled, self.lp, self.ws_d,
                        self.mode)
        L.bi_decode_advance(self.sampled, self.lp, self.tok, self.pos, self.B, self.step, self.hist_ids, self.hist_lp,
                            self.n_gen)

    def _prefill(self, seqs_tokens_dev, cu, cache, targets, logit_from, lp, sm, ws):
        B = self.B
        L.bi_forward_prefill(self.dec.handle, seqs_tokens_dev, targets, cu, [0] * B, logit_from, B, self.chunk,
                             self.bt, self.bt.shape[1], cache.k, cache.v, cache.n_blocks, lp, sm, ws, self.max_tokens,
                             self.max_ctx, self.max_logit_rows, self.mode)

    def rollout(self, prompt_tokens_dev):
        self._prefill(prompt_tokens_dev, self.cu_p, self.cache, None, [int(n) - 1 for n in self.lens], self.lp_p,
                      self.sm_p, self.ws_p)
        self.hist_ids[0] = self.sm_p[self.last]
        self.hist_lp[0] = self.lp_p[self.last]
        self.tok.copy_(self.hist_ids[0])
        self.pos.copy_(self.pos0)
        self.step.fill_(1)
        if self.n_gen <= 1:
            return
        if self.graph is None:
            self._decode_step()       # eager first step, then capture the rest once
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                self._decode_step()
            self.graph = g
            for _ in range(self.n_gen - 2):
                self.graph.replay()
        else:
            for _ in range(self.n_gen - 1):
                self.graph.replay()

    def recompute(self, prompt_tokens_dev):
        self.rec_tok[self.p_dst] = prompt_tokens_dev
        if self.g_dst is not None:
            self.rec_tok[self.g_dst] = self.hist_ids[:-1].T
        self.rec_tgt[self.t_dst] = self.hist_ids.T
        self._prefill(self.rec_tok, self.cu_r, self.cache_r, self.rec_tgt, [int(n) - 1 for n in self.lens],
                      self.rec_lp, None, self.ws_p)
        return self.rec_lp[self.t_dst]

    def run(self, prompt_tokens_dev):
        """Rollout + recompute.  Returns (ids [B, n_gen], rollout lp [B, n_gen], recompute lp [B, n_gen])."""
        self.rollout(prompt_tokens_dev)
        rec = self.recompute(prompt_tokens_dev)
        return self.hist_ids.T, self.hist_lp.T, rec
