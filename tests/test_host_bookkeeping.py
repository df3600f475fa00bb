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
