"""bi_attention_static_scratch: attention for callers that cannot allocate device memory.

Some callers cannot give the library a workspace (hot paths where allocation is
forbidden after start-up, allocators owned by another framework, host
applications that give a plugin no scratch buffer).  For them the library keeps
the attention split partials in a fixed array of its own.  This test calls that
entry point through the C ABI twice in a row, on two different problems (the
second one finds the first one's partials still in the array), and checks each
result against the ordinary workspace entry point; it also checks that a call
too large for the array is refused with a clear error (that check runs on the
host before any CUDA call, and is tested on the CPU in test_abi.py, so that a
regression shows up as a wrong status rather than an out-of-bounds launch).
Decode-shaped calls take the other two schedules (one CTA per split for short
contexts, the persistent one beyond four splits) and BI_FAST takes smaller
splits, i.e. more partials; each is compared with a caller workspace too.  The
file is named so that pytest collects it last.
"""
import math

import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from synthetic import normal_bf16
from tests.gpu_util import dev_bf16, same_bits

pytestmark = pytest.mark.gpu

MAX_POS = 4096


def _problem(seq_lens, Hq, Hkv, hd, seed):
    """A paged cache filled through bi_rope_kv_write and the rotated queries of every row."""
    rng = np.random.default_rng(seed)
    max_blk = max(math.ceil(n / 64) for n in seq_lens)
    n_blocks = len(seq_lens) * max_blk + 2
    bt = torch.from_numpy(rng.permutation(n_blocks)[: len(seq_lens) * max_blk].astype(np.int32)
                          .reshape(len(seq_lens), max_blk)).cuda()
    kc = torch.zeros((n_blocks, Hkv, 64, hd), dtype=torch.bfloat16, device="cuda")
    vc = torch.zeros_like(kc)
    table = torch.empty((MAX_POS, hd), dtype=torch.float32, device="cuda")
    bi.bi_rope_table(table, MAX_POS, hd, 10000.0)
    T = sum(seq_lens)
    qkv = dev_bf16(normal_bf16(rng, (T, (Hq + 2 * Hkv) * hd), 1.0))
    seq = torch.arange(len(seq_lens), dtype=torch.int32, device="cuda")
    row0 = torch.tensor(np.concatenate([[0], np.cumsum(seq_lens)]), dtype=torch.int32, device="cuda")
    pos0 = torch.zeros(len(seq_lens), dtype=torch.int32, device="cuda")
    q = torch.empty((T, Hq, hd), dtype=torch.bfloat16, device="cuda")
    bi.bi_rope_kv_write(qkv, T, seq, row0, pos0, len(seq_lens), max(seq_lens), Hq, Hkv, hd, table, MAX_POS, bt,
                        max_blk, n_blocks, q, kc, vc)
    return dict(q=q, T=T, seq=seq, row0=row0, pos0=pos0, P=len(seq_lens), max_q_len=max(seq_lens), Hq=Hq, Hkv=Hkv,
                hd=hd, kc=kc, vc=vc, bt=bt, max_blk=max_blk, max_ctx=max(seq_lens))


def _decode_rows(pb, seq_lens, pos):
    """Single-token pieces at position `pos` of every sequence longer than it (a decode step)."""
    keep = [b for b, n in enumerate(seq_lens) if pos < n]
    offs = np.concatenate([[0], np.cumsum(seq_lens)])
    rows = torch.tensor([int(offs[b]) + pos for b in keep], device="cuda")
    d = dict(pb)
    d.update(q=pb["q"][rows].contiguous(), T=len(keep), P=len(keep), max_q_len=1,
             seq=torch.tensor(keep, dtype=torch.int32, device="cuda"),
             row0=torch.arange(len(keep) + 1, dtype=torch.int32, device="cuda"),
             pos0=torch.full((len(keep),), pos, dtype=torch.int32, device="cuda"))
    return d


def _with_workspace(pb, mode=bi.BI_INVARIANT):
    out = torch.empty((pb["T"], pb["Hq"] * pb["hd"]), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(bi.bi_attention_workspace_size(pb["T"], pb["Hq"], pb["hd"], pb["max_ctx"], 512),
                     dtype=torch.uint8, device="cuda")
    bi.bi_attention(pb["q"], pb["T"], pb["seq"], pb["row0"], pb["pos0"], pb["P"], pb["max_q_len"], pb["Hq"],
                    pb["Hkv"], pb["hd"], pb["kc"], pb["vc"], pb["bt"], pb["max_blk"], pb["kc"].shape[0],
                    pb["max_ctx"], 512, 1.0 / math.sqrt(pb["hd"]), ws, out, mode)
    return out


def _static(pb, mode=bi.BI_INVARIANT):
    out = torch.full((pb["T"], pb["Hq"] * pb["hd"]), float("nan"), dtype=torch.bfloat16, device="cuda")
    bi.bi_attention_static_scratch(pb["q"], pb["T"], pb["seq"], pb["row0"], pb["pos0"], pb["P"], pb["max_q_len"],
                                   pb["Hq"], pb["Hkv"], pb["hd"], pb["kc"], pb["vc"], pb["bt"], pb["max_blk"],
                                   pb["kc"].shape[0], pb["max_ctx"], 512, 1.0 / math.sqrt(pb["hd"]), out, mode)
    return out


def test_static_scratch_attention_matches_workspace_attention_twice():
    first = _problem([1100, 333, 64, 1], 8, 2, 128, seed=1)    # three splits, GQA 4, 18.7 MB of partials
    second = _problem([700, 5], 8, 8, 64, seed=2)              # smaller problem over stale partials
    want1, want2 = _with_workspace(first), _with_workspace(second)
    got1 = _static(first)
    got2 = _static(second)
    torch.cuda.synchronize()
    # the tolerance of the attention tests is bit equality between two launches of the same kernels
    assert same_bits(got1, want1)
    assert same_bits(got2, want2)
    assert bi.bi_device_status() == 0


def test_static_scratch_decode_schedules_and_fast_mode_match_workspace():
    lens = [3000, 2600, 700, 1]
    pb = _problem(lens, 16, 4, 128, seed=4)
    short = dict(_decode_rows(pb, lens, 650), max_ctx=2048)    # <= 4 splits: one CTA per (seq, kv head, split)
    long_ = _decode_rows(pb, lens, 2999)                       # 6 splits: persistent schedule, TMA page streaming
    for d in (short, long_, short):
        want, got = _with_workspace(d), _static(d)
        torch.cuda.synchronize()
        assert same_bits(got, want)
    # BI_FAST shrinks the split for decode-sized calls (more partials per row)
    want, got = _with_workspace(long_, bi.BI_FAST), _static(long_, bi.BI_FAST)
    torch.cuda.synchronize()
    assert same_bits(got, want)
    assert bi.bi_device_status() == 0
