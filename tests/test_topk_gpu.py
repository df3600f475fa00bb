"""Deterministic Top-K ([Article] §4.3) on the GPU through the C ABI: bit-exact
against the oracle, rows independent of the batch they run in, and the
non-deterministic BI_FAST variant selecting the same scores.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own."""
import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from oracle import topk as otk
from synthetic import C5, make_c5_prompt_lengths

pytestmark = pytest.mark.gpu


def _scores(rng, T, ld, dist):
    if dist == "normal":
        return rng.standard_normal((T, ld)).astype(np.float32)
    if dist == "bf16_ties":   # indexer scores at bf16 precision: frequent exact ties
        s = rng.standard_normal((T, ld)).astype(np.float32)
        return (s.view(np.uint32) & 0xFFFF0000).view(np.float32)
    if dist == "coarse":      # a handful of values, both signed zeros, infinities
        s = rng.integers(-3, 4, (T, ld)).astype(np.float32)
        z = s == 0
        s[z] = np.where(rng.random(z.sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
        s[rng.random((T, ld)) < 0.01] = np.inf
        s[rng.random((T, ld)) < 0.01] = -np.inf
        return s
    return (-np.abs(rng.standard_normal((T, ld))) - 1.0).astype(np.float32)


def _run(S, n_valid, K, mode=bi.BI_INVARIANT):
    T, ld = S.shape
    out = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    bi.bi_topk(torch.from_numpy(S).cuda(), T, ld, torch.from_numpy(np.asarray(n_valid, np.int32)).cuda(), K, out,
               mode)
    return out.cpu().numpy()


@pytest.mark.parametrize("dist", ["normal", "bf16_ties", "coarse", "negative"])
@pytest.mark.parametrize("T,ld,K", [(40, 300, 7), (24, 3000, 64), (12, 5000, 2048), (4, 40000, 4096), (6, 2100, 1)])
def test_topk_matches_oracle(dist, T, ld, K):
    rng = np.random.default_rng(T * ld + K + len(dist))
    S = _scores(rng, T, ld, dist)
    n = rng.integers(0, ld + 1, T)
    n[0], n[-1] = ld, min(K, ld)             # a full row and a row of exactly K candidates
    got = _run(S, n, K)
    want = otk.topk(S, n, K)
    assert np.array_equal(got, want)
    assert bi.bi_device_status() == 0


def test_topk_pages_tie_example():
    """The pages' two-way tie example, every case of the golden fixture in one batch."""
    from tests.test_oracle_topk_pins import golden_tie_cases
    cases = golden_tie_cases()
    ld = max(len(c[0]) for c in cases)
    K = max(c[2] for c in cases)
    S = np.full((len(cases), ld), -1.0, np.float32)
    for t, (s, n, k, want) in enumerate(cases):
        S[t, :len(s)] = s
    n = np.array([c[1] for c in cases])
    for t, (s, nv, k, want) in enumerate(cases):
        got = _run(S[t:t + 1], n[t:t + 1], k)
        assert got[0].tolist() == want, (t, got[0].tolist(), want)
    assert bi.bi_device_status() == 0


def test_topk_edge_rows():
    S = np.full((5, 4096), 0.5, np.float32)
    n = np.array([0, 1, 4096, 2047, 2048])
    got = _run(S, n, 2048)
    assert np.array_equal(got, otk.topk(S, n, 2048))
    assert got[2, :3].tolist() == [4095, 4094, 4093]        # equal scores: the largest positions
    assert (got[0] == -1).all() and got[1, 0] == 0 and (got[1, 1:] == -1).all()


def test_topk_decode_workload_sampled_rows_and_batch_independence():
    """64 rows with the long-context decoder's contexts (1K-32K) and K = 2048 (the
    pages' indexer budget): sampled rows match the oracle; every row is bitwise the
    same run alone, in a shuffled batch, or next to other rows."""
    lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
    rng = np.random.default_rng(17)
    T, ld, K = len(lens), int(lens.max()), 2048
    S = _scores(rng, T, ld, "bf16_ties")
    full = _run(S, lens, K)
    for t in rng.choice(T, 4, replace=False):
        assert np.array_equal(full[t], otk.topk_row(S[t], int(lens[t]), K)), t
    perm = rng.permutation(T)
    assert np.array_equal(_run(S[perm], lens[perm], K), full[perm])
    for t in (0, 17, 63):
        assert np.array_equal(_run(S[t:t + 1], lens[t:t + 1], K), full[t:t + 1])


def test_topk_fast_selects_the_same_scores():
    rng = np.random.default_rng(5)
    T, ld, K = 16, 6000, 512
    S = _scores(rng, T, ld, "coarse")
    n = rng.integers(K + 1, ld + 1, T)
    inv = _run(S, n, K)
    fast = _run(S, n, K, bi.BI_FAST)
    for t in range(T):
        # the same multiset of scores (compared as numbers: -0 == +0), possibly other tie positions
        assert np.array_equal(np.sort(S[t][inv[t]]), np.sort(S[t][fast[t]]))
        assert len(set(fast[t].tolist())) == K and fast[t].min() >= 0 and fast[t].max() < n[t]


def test_topk_row_and_cluster_schedules_agree():
    """400 rows take one CTA per row, 64 or fewer a cluster per row: every row is
    bitwise the same either way, and both equal the oracle."""
    rng = np.random.default_rng(23)
    T, ld, K = 400, 3000, 256
    S = _scores(rng, T, ld, "bf16_ties")
    n = rng.integers(0, ld + 1, T)
    full = _run(S, n, K)
    assert np.array_equal(full, otk.topk(S, n, K))
    for a in (0, 150, 336):
        assert np.array_equal(_run(S[a:a + 64], n[a:a + 64], K), full[a:a + 64])
    fast = _run(S, n, K, bi.BI_FAST)
    for t in range(0, T, 37):
        assert np.array_equal(np.sort(S[t][full[t][full[t] >= 0]]), np.sort(S[t][fast[t][fast[t] >= 0]]))


@pytest.mark.parametrize("dist", ["normal", "coarse", "bf16_ties"])
def test_topk_row_kernel_long_rows(dist):
    """One CTA per row over 32K-position rows: the kept-candidate passes (normal
    scores: the first byte's candidates fit in shared memory) and the full-row
    fallback (coarse scores: most keys share a byte) both give the oracle's result."""
    rng = np.random.default_rng(len(dist) + 99)
    T, ld, K = 320, 32768, 2048
    S = _scores(rng, T, ld, dist)
    n = rng.integers(K, ld + 1, T)
    n[:3] = [ld, K, K + 1]
    got = _run(S, n, K)
    rows = np.r_[0:3, rng.choice(np.arange(3, T), 29, replace=False)]
    assert np.array_equal(got[rows], otk.topk(S[rows], n[rows], K))
    assert bi.bi_device_status() == 0
