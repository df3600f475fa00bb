"""Long-context attention against the oracle: contexts of 4K, 16K and 33K positions.

"vLLM Achieves Bitwise-Consistent RL Training ..." §4.2 puts prefill, decode and
training on one read path with a fixed split (the zero-mismatch-rl README calls it
"fixed-split attention").  The other attention tests show that the schedules agree
with each other bit for bit; this one shows that what they agree on is the
attention itself, deep into contexts of up to 65 splits of 512 (the long-context
workload's 1K-32K prompts plus generated tokens), for:
  * the persistent decode schedule (TMA page streaming, at most 1024 pieces);
  * the per-CTA decode schedule (taken by calls of more than 1024 pieces);
  * the row-parallel prefill schedule, on a 2048-row chunk at positions
    30720..32767 of the longest sequence.
A few sampled rows of each call are compared element by element with the oracle's
explicit softmax over every earlier position (bounds of the short-context
attention parity test: max 2e-2, mean 2e-3).  Cache slots past each sequence's
last position hold NaN.
"""
import math

import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from oracle import ops
from synthetic import bits_to_f32, normal_bf16
from tests.gpu_util import dev_bf16, host_f32, same_bits

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

HQ, HKV, HD = 16, 4, 128
LENS = [4100, 16450, 32900]          # 9, 33 and 65 splits of 512
SPLIT = 512
MAX_POS = 33024


def _pieces(pieces):
    seq = torch.tensor([p[0] for p in pieces], dtype=torch.int32, device="cuda")
    row0 = torch.tensor(np.concatenate([[0], np.cumsum([p[2] for p in pieces])]), dtype=torch.int32, device="cuda")
    pos0 = torch.tensor([p[1] for p in pieces], dtype=torch.int32, device="cuda")
    return seq, row0, pos0


@pytest.fixture(scope="module")
def setup():
    rng = np.random.default_rng(4242)
    max_blk = max(math.ceil(n / 64) for n in LENS)
    n_blocks = len(LENS) * max_blk + 3
    bt = torch.from_numpy(rng.permutation(n_blocks)[: len(LENS) * max_blk].astype(np.int32)
                          .reshape(len(LENS), max_blk)).cuda()
    kc = torch.full((n_blocks, HKV, 64, HD), float("nan"), dtype=torch.bfloat16, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    table = torch.empty((MAX_POS, HD), dtype=torch.float32, device="cuda")
    bi.bi_rope_table(table, MAX_POS, HD, 10000.0)
    T = sum(LENS)
    qkv_bits = normal_bf16(rng, (T, (HQ + 2 * HKV) * HD), 1.0)
    qkv = dev_bf16(qkv_bits)
    seq, row0, pos0 = _pieces([(b, 0, n) for b, n in enumerate(LENS)])
    q = torch.empty((T, HQ, HD), dtype=torch.bfloat16, device="cuda")
    bi.bi_rope_kv_write(qkv, T, seq, row0, pos0, len(LENS), max(LENS), HQ, HKV, HD, table, MAX_POS, bt, max_blk,
                        n_blocks, q, kc, vc)
    torch.cuda.synchronize()
    # the oracle's own q, k, v (RoPE from the same bf16 inputs, not from the GPU's cache)
    f = bits_to_f32(qkv_bits)
    offs = np.concatenate([[0], np.cumsum(LENS)])
    oq, ok, ov = [], [], []
    for b, n in enumerate(LENS):
        fb = f[offs[b]:offs[b + 1]]
        pos = np.arange(n)
        oq.append(ops.rope(fb[:, : HQ * HD].reshape(n, HQ, HD), pos))
        ok.append(ops.rope(fb[:, HQ * HD:(HQ + HKV) * HD].reshape(n, HKV, HD), pos))
        ov.append(fb[:, (HQ + HKV) * HD:].reshape(n, HKV, HD))
    return dict(bt=bt, kc=kc, vc=vc, q=q, offs=offs, max_blk=max_blk, n_blocks=n_blocks, oq=oq, ok=ok, ov=ov)


def _attend(s, pieces, rows, max_q_len, max_ctx):
    """bi_attention over `pieces` whose query rows are the prefill q rows `rows`."""
    seq, row0, pos0 = _pieces(pieces)
    T = len(rows)
    q = s["q"][torch.as_tensor(np.asarray(rows), device="cuda")].contiguous()
    out = torch.empty((T, HQ * HD), dtype=torch.bfloat16, device="cuda")
    ns = -(-max_ctx // SPLIT)
    ws = torch.empty(T * HQ * ns * (HD + 2) * 4 + 256, dtype=torch.uint8, device="cuda")
    bi.bi_attention(q, T, seq, row0, pos0, len(pieces), max_q_len, HQ, HKV, HD, s["kc"], s["vc"], s["bt"],
                    s["max_blk"], s["n_blocks"], max_ctx, SPLIT, 1.0 / math.sqrt(HD), ws, out)
    torch.cuda.synchronize()
    return host_f32(out)


def _oracle_row(s, b, p):
    """The oracle's attention output of sequence b's row at position p (explicit softmax)."""
    return ops.attention(s["oq"][b][p:p + 1], s["ok"][b][:p + 1], s["ov"][b][:p + 1], np.array([p])).reshape(-1)


def _check(got_rows, want_rows):
    err = np.abs(np.asarray(got_rows) - np.asarray(want_rows))
    assert np.isfinite(got_rows).all()
    assert err.max() < 2e-2 and err.mean() < 2e-3, (err.max(), err.mean())
    return err


def _decode_pieces(n_pieces, seed):
    """n_pieces single-token decode rows at seeded positions of the three sequences,
    always including each sequence's last position and a split boundary."""
    rng = np.random.default_rng(seed)
    pcs = [(b, n - 1, 1) for b, n in enumerate(LENS)] + [(2, 512 * 40, 1), (2, 512 * 40 - 1, 1)]
    while len(pcs) < n_pieces:
        b = int(rng.integers(0, len(LENS)))
        pcs.append((b, int(rng.integers(0, LENS[b])), 1))
    order = rng.permutation(len(pcs))
    return [pcs[i] for i in order]


def test_long_context_decode_schedules_match_the_oracle(setup):
    s = setup
    max_ctx = max(LENS)
    pcs_p = _decode_pieces(1000, seed=1)              # persistent schedule (<= 1024 pieces)
    pcs_c = pcs_p + _decode_pieces(100, seed=2)       # per-CTA schedule (> 1024 pieces)
    rows_p = [int(s["offs"][b]) + p for b, p, _ in pcs_p]
    rows_c = [int(s["offs"][b]) + p for b, p, _ in pcs_c]
    got_p = _attend(s, pcs_p, rows_p, 1, max_ctx)
    got_c = _attend(s, pcs_c, rows_c, 1, max_ctx)
    # both schedules give the same bits on the rows they share
    assert np.array_equal(got_p.view(np.uint32), got_c[: len(pcs_p)].view(np.uint32))
    # and those bits are the attention: the last row of each sequence, the split
    # boundary rows and a few seeded ones, against the oracle
    pick = [i for i, (b, p, _) in enumerate(pcs_c) if p == LENS[b] - 1 or p in (512 * 40, 512 * 40 - 1)]
    pick += list(np.random.default_rng(3).choice(len(pcs_c), 6, replace=False))
    for i in sorted(set(pick)):
        b, p, _ = pcs_c[i]
        _check(got_c[i], _oracle_row(s, b, p))


def test_long_context_prefill_chunk_deep_in_the_context_matches_the_oracle(setup):
    s = setup
    b, p0, ch = 2, 30720, 2048
    rows = list(range(int(s["offs"][b]) + p0, int(s["offs"][b]) + p0 + ch))
    got = _attend(s, [(b, p0, ch)], rows, ch, max(LENS))
    for r in (0, 1, 511, 1024, 2047) + tuple(np.random.default_rng(4).integers(0, ch, 3)):
        _check(got[r], _oracle_row(s, b, p0 + int(r)))
    # the same rows as single-token decode rows are bit-equal to the chunk's rows
    pcs = [(b, p0 + r, 1) for r in (0, 777, 2047)]
    dec = _attend(s, pcs, [rows[0], rows[777], rows[2047]], 1, max(LENS))
    assert np.array_equal(dec.view(np.uint32), got[[0, 777, 2047]].view(np.uint32))
    assert bi.bi_device_status() == 0
