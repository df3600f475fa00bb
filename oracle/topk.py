"""Deterministic Top-K oracle (test infrastructure only).

[Article] §4.3, "Top-K in sparse attention: fix ties and order".  Every
candidate of a row is a pair (score, in-request position).  The K candidates
that come first in the order "higher score first, and between equal scores the
larger position first" are selected (the pages combine score and position into
one unique key so that ties go to the larger position), and the selected
positions are written in descending position order, invalid entries (-1) last
when the row has fewer than K candidates.

Readings where the pages are silent:
  * Candidates of a row are the positions 0 .. n_valid - 1 (the in-request
    positions; nothing else of the batch enters the key).
  * Scores compare as real numbers: -0.0 and +0.0 are equal (a tie, decided by
    position); -inf is a score like any other.  NaN is outside the contract.

The selection is written directly from that definition: a stable sort of the
candidates by (score desc, position desc), take K, sort the positions
descending.  Nothing here is blocked, fused or reordered.

[Article] is "vLLM Achieves Bitwise-Consistent RL Training: Eliminating Numerical
Drift to Zero KL Divergence on DeepSeek-V4-Flash at 91% Throughput"; section numbers
are its own.
"""
from __future__ import annotations

import numpy as np


def topk_row(scores, n_valid: int, k: int) -> np.ndarray:
    """Selected positions of one row, descending, padded with -1 to length k."""
    s = np.asarray(scores, dtype=np.float32)[:n_valid]
    cand = sorted(range(n_valid), key=lambda p: (-float(s[p]), -p))   # score desc, then position desc
    chosen = sorted(cand[:k], reverse=True)
    return np.array(chosen + [-1] * (k - len(chosen)), dtype=np.int32)


def topk(scores, n_valid, k: int) -> np.ndarray:
    """Rows of scores [T, ld] (fp32) with per-row candidate counts n_valid [T] -> int32 [T, k]."""
    scores = np.asarray(scores, dtype=np.float32)
    return np.stack([topk_row(scores[t], int(n_valid[t]), k) for t in range(scores.shape[0])]).astype(np.int32)
