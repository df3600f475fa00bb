"""Pins of the deterministic Top-K oracle ([Article] §4.3) against things other than itself:
the pages' own two-way tie example, closed forms, brute force on tiny rows, and an
independent restatement through the 64-bit (score, position) key the pages describe.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own."""
import itertools
import json
import os

import numpy as np
import pytest

from oracle import topk as otk


def _ordered_u32(x: np.ndarray) -> np.ndarray:
    """Order-preserving map of fp32 to uint32 (after -0 -> +0): larger float, larger integer."""
    x = np.where(x == 0, np.float32(0), x).astype(np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    return np.where(u >> 31, (~u) & 0xFFFFFFFF, u | 0x80000000).astype(np.uint64)


def _topk_by_key(scores, n, k):
    """The pages' formulation: key = score bits << 32 | position, K largest keys, positions descending."""
    s = np.asarray(scores, np.float32)[:n]
    key = (_ordered_u32(s) << np.uint64(32)) | np.arange(n, dtype=np.uint64)
    top = np.sort(key)[::-1][:k]
    pos = np.sort((top & np.uint64(0xFFFFFFFF)).astype(np.int64))[::-1]
    return np.concatenate([pos, -np.ones(k - len(pos), np.int64)]).astype(np.int32)


def golden_tie_cases():
    """The pages' two-way tie example (tests/golden/topk_tie_example.json, with its
    citation): (scores, n_valid, k, want) per case."""
    with open(os.path.join(os.path.dirname(__file__), "golden", "topk_tie_example.json")) as f:
        g = json.load(f)
    out = []
    for c in g["cases"]:
        s = np.full(max(64, c["n_valid"]), c["default"], np.float32)
        for p, v in c["scores"].items():
            s[int(p)] = v
        out.append((s, c["n_valid"], c["k"], c["want"]))
    return out


def test_pages_tie_example_selects_larger_position():
    # K = 2; positions 17 and 42 tie: the position bits select 42, and the output
    # lists selected positions by descending position, invalid entries last
    cases = golden_tie_cases()
    assert len(cases) >= 2 and cases[0][3] == [42, 5]
    for s, n, k, want in cases:
        assert otk.topk_row(s, n, k).tolist() == want, (n, k)
        assert _topk_by_key(s, n, k).tolist() == want, (n, k)


def test_fewer_candidates_than_k_pads_with_invalid_last():
    s = np.array([0.5, 2.0, -1.0, 7.0], np.float32)
    assert otk.topk_row(s, 3, 5).tolist() == [2, 1, 0, -1, -1]
    assert otk.topk_row(s, 0, 2).tolist() == [-1, -1]


def test_all_equal_scores_take_the_largest_positions():
    s = np.full(100, 0.25, np.float32)
    assert otk.topk_row(s, 100, 4).tolist() == [99, 98, 97, 96]


def test_signed_zeros_tie_and_infinities_order():
    s = np.array([1.0, 0.0, -3.0, -0.0, -np.inf, np.inf], np.float32)
    assert otk.topk_row(s, 6, 1).tolist() == [5]             # +inf first
    assert otk.topk_row(s, 6, 3).tolist() == [5, 3, 0]       # -0.0 ties +0.0; position 3 > 1
    assert otk.topk_row(s, 6, 6).tolist() == [5, 4, 3, 2, 1, 0]
    assert otk.topk_row(s[:5], 5, 5).tolist() == [4, 3, 2, 1, 0]


def test_bruteforce_tiny_rows():
    rng = np.random.default_rng(3)
    for _ in range(200):
        n = int(rng.integers(1, 8))
        k = int(rng.integers(1, 8))
        s = rng.integers(-2, 3, n).astype(np.float32)          # many exact ties
        got = otk.topk_row(s, n, k)
        sel = [p for p in got.tolist() if p >= 0]
        assert len(sel) == min(n, k) and sel == sorted(sel, reverse=True)
        # every chosen candidate beats every other one in (score, position) order
        rest = [p for p in range(n) if p not in sel]
        for a, b in itertools.product(sel, rest):
            assert (s[a], a) > (s[b], b)


@pytest.mark.parametrize("dist", ["normal", "bf16_ties", "negative", "coarse"])
def test_matches_64bit_key_restatement(dist):
    rng = np.random.default_rng(len(dist))
    T, ld = 24, 700
    if dist == "normal":
        S = rng.standard_normal((T, ld)).astype(np.float32)
    elif dist == "bf16_ties":
        S = rng.standard_normal((T, ld)).astype(np.float32)
        S = (S.view(np.uint32) & 0xFFFF0000).view(np.float32)    # truncate to bf16: frequent exact ties
    elif dist == "negative":
        S = -np.abs(rng.standard_normal((T, ld))).astype(np.float32) - 1.0
    else:
        S = rng.integers(-3, 4, (T, ld)).astype(np.float32)
        S[S == 0] = np.where(rng.random((S == 0).sum()) < 0.5, np.float32(0.0), np.float32(-0.0))
    n_valid = rng.integers(0, ld + 1, T)
    for k in (1, 7, 64, 512):
        got = otk.topk(S, n_valid, k)
        for t in range(T):
            assert np.array_equal(got[t], _topk_by_key(S[t], int(n_valid[t]), k)), (dist, k, t)


def test_rows_are_independent():
    rng = np.random.default_rng(9)
    S = rng.standard_normal((6, 50)).astype(np.float32)
    n = np.array([50, 10, 0, 49, 1, 33])
    full = otk.topk(S, n, 8)
    perm = rng.permutation(6)
    assert np.array_equal(otk.topk(S[perm], n[perm], 8), full[perm])
