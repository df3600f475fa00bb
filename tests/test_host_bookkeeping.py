"""Host bookkeeping of the rollout / recompute driver, on the CPU: block tables
and the training side's packed batch (prompt + response, targets and scored
rows) in its two forms, the list form of `Decoder.recompute` and the static
row indices of `Episode`."""
import numpy as np

from invariant_forward_policy_gb300.decoder import block_ids, paged_block_ids, recompute_pack, recompute_rows


def test_block_ids_are_a_permutation_of_the_range():
    t = block_ids(5, 7, seed=3, base=10)
    assert t.shape == (5, 7) and t.dtype == np.int32
    assert sorted(t.ravel().tolist()) == list(range(10, 45))
    assert np.array_equal(block_ids(5, 7, seed=3, base=10), t)              # seeded
    assert not np.array_equal(block_ids(5, 7, seed=4, base=10), t)
    assert np.array_equal(block_ids(2, 3), np.arange(6, dtype=np.int32).reshape(2, 3))


def test_paged_block_ids_give_each_context_its_own_blocks():
    lens = [1, 64, 65, 0, 300, 128]
    tab, total = paged_block_ids(lens, 6, seed=9)
    need = [1, 1, 2, 0, 5, 2]
    assert total == sum(need) and tab.shape == (6, 6)
    used = []
    for b, n in enumerate(need):
        assert (tab[b, n:] == -1).all() and (tab[b, :n] >= 0).all()
        used += tab[b, :n].tolist()
    assert sorted(used) == list(range(total))                                 # disjoint, all used


def _random_batch(rng, B, n_gen):
    prompts = [rng.integers(0, 1000, int(rng.integers(1, 40))).astype(np.int32) for _ in range(B)]
    gens = [rng.integers(0, 1000, n_gen).astype(np.int32) for _ in range(B)]
    return prompts, gens


def test_recompute_pack_feeds_back_all_but_the_last_token():
    rng = np.random.default_rng(1)
    prompts, gens = _random_batch(rng, 4, 6)
    order = [2, 0, 3, 1]
    seqs, tg, lf = recompute_pack(prompts, gens, order)
    for j, b in enumerate(order):
        p, g = prompts[b], gens[b]
        assert np.array_equal(seqs[j], np.concatenate([p, g[:-1]]))
        assert lf[j] == len(p) - 1
        # row r's target is the token that follows it: the next prompt token is not
        # scored (target 0), and rows len(p) - 1 .. predict the generated tokens
        assert np.array_equal(tg[j][lf[j]:], g) and (tg[j][:lf[j]] == 0).all()
        assert np.array_equal(tg[j][lf[j]:-1], seqs[j][lf[j] + 1:])


def test_static_rows_build_the_same_batch_as_the_list_form():
    rng = np.random.default_rng(2)
    for n_gen in (1, 2, 9):
        prompts, gens = _random_batch(rng, 5, n_gen)
        cu, p_dst, g_dst, t_dst = recompute_rows([len(p) for p in prompts], n_gen)
        seqs, tg, lf = recompute_pack(prompts, gens, range(5))
        assert cu[-1] == sum(len(s) for s in seqs) and np.array_equal(np.diff(cu), [len(s) for s in seqs])
        tok = np.full(int(cu[-1]), -1, np.int64)
        tgt = np.zeros(int(cu[-1]), np.int64)
        tok[p_dst] = np.concatenate(prompts)
        G = np.stack(gens)
        if n_gen > 1:
            assert g_dst.shape == (5, n_gen - 1)
            tok[g_dst] = G[:, :-1]
        else:
            assert g_dst is None
        tgt[t_dst] = G
        assert np.array_equal(tok, np.concatenate(seqs))                      # every row written once
        assert np.array_equal(tgt, np.concatenate(tg))
        assert np.array_equal(t_dst[:, 0], cu[:-1] + np.array(lf))


def _check_plan(lens, start_pos, logit_from, chunk, max_tokens):
    from invariant_forward_policy_gb300 import bi_prefill_plan
    B = len(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    plan = bi_prefill_plan(cu.tolist(), list(start_pos), None if logit_from is None else list(logit_from), chunk,
                           max_tokens)
    seen = [0] * B                        # rows of each sequence scheduled so far
    logits = [0] * B
    passes = {}
    last_chunk = -1
    for p, seq, row0, rows, pos0, tok0, lfirst, loff in plan:
        off = seen[seq]
        assert rows >= 1 and tok0 == cu[seq] + off and pos0 == start_pos[seq] + off   # in order, no gap, no repeat
        assert off // chunk == (off + rows - 1) // chunk and rows <= chunk              # inside one chunk
        assert off // chunk >= last_chunk - 1                                          # chunk-major order
        last_chunk = max(last_chunk, off // chunk)
        lf = 0 if logit_from is None else logit_from[seq]
        assert lfirst == min(max(lf - off, 0), rows)
        seen[seq] += rows
        logits[seq] += rows - lfirst
        passes.setdefault(p, []).append((row0, rows, lfirst, loff))
    assert seen == list(lens)                                                          # every row once
    for b in range(B):
        lf = 0 if logit_from is None else logit_from[b]
        assert logits[b] == lens[b] - min(max(lf, 0), lens[b])
    assert sorted(passes) == list(range(len(passes)))
    for pieces in passes.values():
        assert len(pieces) <= min(128, max(B, 1))
        r = lo = 0
        for row0, rows, lfirst, loff in pieces:                                         # packed back to back
            assert row0 == r and loff == lo
            r += rows
            lo += rows - lfirst
        assert r <= max_tokens
    return plan


def test_prefill_plan_schedules_every_row_once_within_the_limits():
    rng = np.random.default_rng(3)
    for trial in range(300):
        B = int(rng.integers(1, 200 if trial % 7 == 0 else 10))
        lens = rng.integers(0, 2500, B)
        sp = rng.integers(0, 300, B)
        lf = (rng.integers(0, 2500, B) * rng.integers(0, 2, B)) if trial % 2 else None
        chunk = int(rng.choice([1, 64, 97, 512, 2048, 1 << 30]))
        mt = int(rng.choice([3, 64, 500, 2048, 8192]))
        _check_plan(lens, sp, lf, chunk, mt)


def test_prefill_plan_small_cases_and_errors():
    import pytest
    import invariant_forward_policy_gb300 as bi
    # two sequences, chunk 4, passes of at most 6 rows filled greedily in chunk-major
    # order: chunk 0 of each (4 + 4 > 6: two passes), then chunk 1 of each
    plan = _check_plan([6, 5], [0, 10], None, 4, 6)
    assert [(p, s, r) for p, s, _, r, *_ in plan] == [(0, 0, 4), (1, 1, 4), (1, 0, 2), (2, 1, 1)]
    assert plan[1][4] == 10 and plan[3][4] == 14                                          # positions follow start_pos
    # a piece longer than a pass is split across passes
    plan = _check_plan([10], [0], None, 1 << 20, 4)
    assert [r for _, _, _, r, *_ in plan] == [4, 4, 2]
    assert bi.bi_prefill_plan([0], [], None, 64, 64) == []                                 # no sequences
    with pytest.raises(bi.BiError):
        bi.bi_prefill_plan([1, 5], [0], None, 64, 64)                                      # cu_seqlens[0] != 0
    with pytest.raises(bi.BiError):
        bi.bi_prefill_plan([0, 5, 3], [0, 0], None, 64, 64)                                # decreasing
