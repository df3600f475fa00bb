"""The seeded input generators produce what the input recipe states: shapes, value
distributions, length mixes, bf16-exact values and reproducibility by seed."""
import math

import numpy as np

from synthetic import (C1, C2, C3, C4, C5, DecoderShape, bits_to_f32, make_c5_prompt_lengths, make_decoder_weights,
                       make_logprob_head, make_moe_layer, make_prompts, normal_bf16, to_bf16_bits)


def test_workload_table():
    assert C2["shape"] == DecoderShape(4, 512, 8, 8, 64, 1408, 32000)
    assert (C2["batch"], C2["prompt_min"], C2["prompt_max"], C2["gen"], C2["seed"]) == (16, 128, 512, 256, 202)
    assert C5["shape"] == DecoderShape(8, 2048, 16, 4, 128, 5632, 32000)
    assert (C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["chunk"], C5["seed"]) == (64, 1024, 32768, 2048, 505)
    assert (C1["n_seq"] * C1["seq_len"], C1["d"], C1["vocab"], C1["seed"]) == (512, 256, 4096, 101)
    assert (C3["n_tokens"], C3["d"], C3["ffn"], C3["n_experts"], C3["top_k"], C3["seed"]) == (4096, 2048, 1024, 64, 8, 303)
    assert (C4["n_tokens"], C4["d"], C4["vocab"], C4["w_std"], C4["seed"]) == (16384, 4096, 129280, 0.01, 404)
    for c in (C2["shape"], C5["shape"]):
        assert c.kv_block == 64 and c.kv_split == 512 and c.eps == 1e-6 and c.rope_theta == 10000.0


def test_bf16_normals_are_exact_bf16_with_the_stated_std():
    rng = np.random.default_rng(0)
    b = normal_bf16(rng, (200000,), 0.02)
    x = bits_to_f32(b)
    assert np.array_equal(to_bf16_bits(x), b)                        # every value is a bf16 value
    assert abs(float(x.mean())) < 3 * 0.02 / math.sqrt(x.size)
    assert abs(float(x.std()) / 0.02 - 1.0) < 0.01
    assert np.array_equal(normal_bf16(np.random.default_rng(0), (200000,), 0.02), b)    # seeded


def test_prompt_lengths_and_ids():
    p = make_prompts(C2["batch"], C2["prompt_min"], C2["prompt_max"], C2["shape"].vocab, C2["seed"])
    lens = np.array([len(x) for x in p])
    assert len(p) == 16 and lens.min() >= 128 and lens.max() <= 512
    ids = np.concatenate(p)
    assert ids.dtype == np.int32 and ids.min() >= 0 and ids.max() < 32000
    big = make_prompts(4000, 128, 512, 32000, 7)
    bl = np.array([len(x) for x in big])
    assert abs(bl.mean() - 320.0) < 4.0 and bl.min() == 128 and bl.max() == 512    # uniform on 128..512
    q = make_prompts(C2["batch"], C2["prompt_min"], C2["prompt_max"], C2["shape"].vocab, C2["seed"])
    assert all(np.array_equal(a, b) for a, b in zip(p, q))


def test_long_context_lengths_are_log_uniform():
    n = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
    assert n.shape == (64,) and n.min() >= 1024 and n.max() <= 32768
    many = make_c5_prompt_lengths(20000, 1024, 32768, 11)
    lg = np.log(many)
    lo, hi = math.log(1024), math.log(32768)
    assert abs(lg.mean() - (lo + hi) / 2) < 0.03
    assert abs(lg.std() - (hi - lo) / math.sqrt(12)) < 0.03                # uniform in the logarithm
    h, _ = np.histogram(lg, bins=5, range=(lo, hi))
    assert h.min() > 0.9 * 20000 / 5


def test_decoder_weight_layout_and_gains():
    s = DecoderShape(2, 64, 4, 2, 16, 96, 300)
    w = make_decoder_weights(s, seed=3)
    assert w["embed"].shape == (300, 64) and w["lm_head"].shape == (300, 64) and w["final_norm"].shape == (64,)
    lw = w["layers"][1]
    assert lw["wqkv"].shape == ((4 + 2 * 2) * 16, 64) and lw["wo"].shape == (64, 64)
    assert lw["w13"].shape == (2 * 96, 64) and lw["w2"].shape == (64, 96)
    assert (bits_to_f32(lw["attn_norm"]) == 1.0).all() and (bits_to_f32(w["final_norm"]) == 1.0).all()
    g = bits_to_f32(make_decoder_weights(s, seed=3, random_gains=True)["layers"][0]["ffn_norm"])
    assert not (g == 1.0).all() and abs(float(g.mean()) - 1.0) < 0.05


def test_head_and_moe_generators():
    hd = make_logprob_head(64, 32, 100, 0.02, seed=5)
    assert hd["h"].shape == (64, 32) and hd["w"].shape == (100, 32) and hd["ids"].max() < 100
    m = make_moe_layer(16, 32, 8, 4, 0.02, seed=6)
    assert m["x"].shape == (16, 32) and m["router_logits"].dtype == np.float32
    assert m["w13"].shape == (4, 16, 32) and m["w2"].shape == (4, 32, 8)
