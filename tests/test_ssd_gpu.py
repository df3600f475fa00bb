"""Mamba-2 chunked scan ([Article] §6) through the C ABI: parity with the sequential
fp64 recurrence, and the same bits for every row whether the sequence runs as one
prefill, as prefill chunks of any size, or token by token as decode.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own."""
import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from oracle import ssd as ossd
from synthetic import bits_to_f32, normal_bf16
from tests.gpu_util import dev_bf16

pytestmark = pytest.mark.gpu

H, G, P, N, Q = 4, 2, 64, 128, 64


def _inputs(rng, lens):
    T = int(sum(lens))
    xb = normal_bf16(rng, (T, H, P), 1.0)
    Bb = normal_bf16(rng, (T, G, N), N ** -0.5)
    Cb = normal_bf16(rng, (T, G, N), N ** -0.5)
    loga = (-np.abs(rng.standard_normal((T, H))) * 0.15).astype(np.float32)
    return xb, Bb, Cb, loga


class Scan:
    """Runs calls of pieces against one state store; collects y per sequence and position."""

    def __init__(self, xb, Bb, Cb, loga, lens):
        self.lens = list(lens)
        self.offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
        self.x, self.B, self.C, self.l = xb, Bb, Cb, loga
        nb = bi.bi_ssd_state_bytes(H, G, P, N, Q)
        self.state = torch.zeros((len(lens), nb // 4), dtype=torch.float32, device="cuda")
        self.y = [np.full((n, H, P), np.nan, np.float32) for n in lens]

    def call(self, pieces):
        """pieces: list of (seq, pos0, n) with at most one piece per sequence."""
        rows = np.concatenate([np.arange(self.offs[s] + p0, self.offs[s] + p0 + n) for s, p0, n in pieces])
        T = len(rows)
        y = torch.empty((T, H, P), dtype=torch.float32, device="cuda")
        seq = torch.tensor([p[0] for p in pieces], dtype=torch.int32, device="cuda")
        row0 = torch.tensor(np.concatenate([[0], np.cumsum([p[2] for p in pieces])]), dtype=torch.int32,
                            device="cuda")
        pos0 = torch.tensor([p[1] for p in pieces], dtype=torch.int32, device="cuda")
        bi.bi_ssd_chunk_scan(dev_bf16(self.x[rows]), dev_bf16(self.B[rows]), dev_bf16(self.C[rows]),
                             torch.from_numpy(self.l[rows]).cuda(), seq, row0, pos0, len(pieces),
                             max(p[2] for p in pieces), H, G, P, N, Q, self.state, len(self.lens), y)
        yh = y.cpu().numpy()
        r = 0
        for s, p0, n in pieces:
            self.y[s][p0:p0 + n] = yh[r:r + n]
            r += n


def _run_chunked(inp, lens, chunk, order=None):
    sc = Scan(*inp, lens)
    progress = [0] * len(lens)
    order = list(range(len(lens))) if order is None else order
    while any(progress[s] < lens[s] for s in order):
        pieces = []
        for s in order:
            if progress[s] < lens[s]:
                n = min(chunk(s, progress[s]), lens[s] - progress[s])
                pieces.append((s, progress[s], n))
                progress[s] += n
        sc.call(pieces)
    return sc


def test_ssd_matches_sequential_recurrence():
    rng = np.random.default_rng(1)
    lens = [200, 64, 1, 130]
    inp = _inputs(rng, lens)
    sc = _run_chunked(inp, lens, lambda s, p: 10 ** 9)        # one prefill call
    xb, Bb, Cb, loga = inp
    for s, n in enumerate(lens):
        r = slice(sc.offs[s], sc.offs[s] + n)
        want, _ = ossd.ssd_scan(bits_to_f32(xb[r]), bits_to_f32(Bb[r]), bits_to_f32(Cb[r]), loga[r], n_groups=G)
        err = np.abs(sc.y[s] - want)
        assert err.max() <= 1e-4 * max(1.0, np.abs(want).max()), (s, err.max())
        assert err.mean() <= 1e-5 * max(1.0, np.abs(want).mean())
    assert bi.bi_device_status() == 0


def test_ssd_decode_replays_prefill_bitwise():
    rng = np.random.default_rng(2)
    lens = [200, 64, 1, 130, 129]
    inp = _inputs(rng, lens)
    full = _run_chunked(inp, lens, lambda s, p: 10 ** 9)
    runs = {
        "decode": _run_chunked(inp, lens, lambda s, p: 1),
        "chunks97": _run_chunked(inp, lens, lambda s, p: 97),
        "chunks37_reversed": _run_chunked(inp, lens, lambda s, p: 37, order=[4, 3, 2, 1, 0]),
        "prompt_then_decode": _run_chunked(inp, lens, lambda s, p: 70 if p == 0 else 1),
        "chunk64": _run_chunked(inp, lens, lambda s, p: 64),
    }
    for name, sc in runs.items():
        for s in range(len(lens)):
            assert np.array_equal(sc.y[s].view(np.uint32), full.y[s].view(np.uint32)), (name, s)
        # the stored state: the state entering the open chunk, and that chunk's
        # inputs so far (slots past them are scratch, never read)
        assert _live_state_equal(sc, full, lens), name


def _live_state_equal(a, b, lens):
    sa, sb = a.state.view(torch.int32).cpu().numpy(), b.state.view(torch.int32).cpu().numpy()
    nh = H * N * P
    for s, n in enumerate(lens):
        k = n % Q
        if not np.array_equal(sa[s, :nh], sb[s, :nh]):
            return False
        for off, width in ((nh, H * N), (nh + Q * H * N, H * P), (nh + Q * H * N + Q * H * P, H)):
            if not np.array_equal(sa[s, off:off + k * width], sb[s, off:off + k * width]):
                return False
    return True


def test_ssd_rows_do_not_depend_on_the_batch():
    rng = np.random.default_rng(3)
    lens = [150, 90, 33]
    inp = _inputs(rng, lens)
    together = _run_chunked(inp, lens, lambda s, p: 50)
    for s in range(len(lens)):
        alone = Scan(*inp, lens)
        p = 0
        while p < lens[s]:
            n = min(50, lens[s] - p)
            alone.call([(s, p, n)])
            p += n
        assert np.array_equal(alone.y[s].view(np.uint32), together.y[s].view(np.uint32)), s


def test_ssd_full_size_sampled_against_recurrence():
    """The timed prefill workload in its launch configuration (16 sequences x 2048
    positions in one call; 32 heads x 64, state 128, 8 groups, chunk 64), sampled
    (sequence, head) pairs against the fp64 recurrence run for that head alone."""
    Hf, Gf, n_seq, per = 32, 8, 16, 2048
    T = n_seq * per
    rng = np.random.default_rng(8)
    xb = normal_bf16(rng, (T, Hf, P), 1.0)
    Bb = normal_bf16(rng, (T, Gf, N), N ** -0.5)
    Cb = normal_bf16(rng, (T, Gf, N), N ** -0.5)
    loga = (-np.abs(rng.standard_normal((T, Hf))) * 0.15).astype(np.float32)
    state = torch.zeros((n_seq, bi.bi_ssd_state_bytes(Hf, Gf, P, N, Q) // 4), dtype=torch.float32, device="cuda")
    y = torch.empty((T, Hf, P), dtype=torch.float32, device="cuda")
    seq = torch.arange(n_seq, dtype=torch.int32, device="cuda")
    row0 = torch.arange(0, T + 1, per, dtype=torch.int32, device="cuda")
    pos0 = torch.zeros(n_seq, dtype=torch.int32, device="cuda")
    bi.bi_ssd_chunk_scan(dev_bf16(xb), dev_bf16(Bb), dev_bf16(Cb), torch.from_numpy(loga).cuda(), seq, row0, pos0,
                         n_seq, per, Hf, Gf, P, N, Q, state, n_seq, y)
    yh = y.cpu().numpy()
    assert np.isfinite(yh).all()
    for s, h in ((0, 0), (7, 13), (15, 31)):
        g = h // (Hf // Gf)
        r = slice(s * per, (s + 1) * per)
        want, _ = ossd.ssd_scan(bits_to_f32(xb[r, h:h + 1]), bits_to_f32(Bb[r, g:g + 1]), bits_to_f32(Cb[r, g:g + 1]),
                                loga[r, h:h + 1], n_groups=1)
        err = np.abs(yh[r, h:h + 1] - want)
        assert err.max() <= 1e-4 * max(1.0, np.abs(want).max()), (s, h, err.max())
        assert err.mean() <= 1e-5 * max(1.0, np.abs(want).mean()), (s, h, err.mean())
    assert bi.bi_device_status() == 0
