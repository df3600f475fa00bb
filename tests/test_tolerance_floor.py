"""The free-running logprob bounds of tests/parity.py rest on a measured noise floor.

For each model the GPU tests score free running, the oracle is compared with
variants of itself that change only what a second implementation of the same
numerical contract may change: the accumulation order (here fp64) and the bf16
rounding of the attention probabilities before P.V (see tests/noise_floor.py).
Every bound must lie between the largest floor measured for its model and
2.5 times it: large enough that a correct kernel passes, small enough that the
bound still means something.  (The 5e-3 target for GPU logprobs against the
oracle sits below the maximum of this floor on every multi-layer model; it is
met as a mean on the dense decoder.)
"""
import numpy as np
import pytest

from oracle import model as omodel
from synthetic import C2, C5, DecoderShape, make_c5_prompt_lengths, make_decoder_weights, make_prompts
from tests import parity
from tests.noise_floor import floors

SLACK = 2.5


def _small():
    # the 2-layer model of the small rollout test (d 128, GQA 4/2, hd 64), 5 prompts, 40 tokens
    shape = DecoderShape(2, 128, 4, 2, 64, 256, 512)
    W = omodel.weights_to_f32(make_decoder_weights(shape, seed=31, w_std=0.05))
    P = make_prompts(5, 10, 150, shape.vocab, seed=32)
    return shape, W, P, 40


def _small_gqa():
    # the 2-layer long-context test model (d 256, GQA 16/4, hd 128), one 500-1500-token prompt
    shape = DecoderShape(2, 256, 16, 4, 128, 512, 1024)
    W = omodel.weights_to_f32(make_decoder_weights(shape, seed=41, w_std=0.05))
    P = make_prompts(4, 500, 1500, shape.vocab, seed=42)[:1]
    return shape, W, P, 24


def _dense():
    # the dense-decoder workload: sequences 0, 5, 10, 15 of 16, 256 tokens each
    shape = C2["shape"]
    W = omodel.weights_to_f32(make_decoder_weights(shape, seed=C2["seed"], w_std=C2["w_std"]))
    prompts = make_prompts(C2["batch"], C2["prompt_min"], C2["prompt_max"], shape.vocab, C2["seed"])
    return shape, W, [prompts[b] for b in (0, 5, 10, 15)], 256


def _long():
    # the long-context GQA workload's shortest sequence (1037 tokens), 64 tokens
    shape = C5["shape"]
    W = omodel.weights_to_f32(make_decoder_weights(shape, seed=C5["seed"], w_std=C5["w_std"]))
    lens = make_c5_prompt_lengths(C5["batch"], C5["ctx_min"], C5["ctx_max"], C5["seed"])
    rng = np.random.default_rng(C5["seed"] + 3)
    prompts = [rng.integers(0, shape.vocab, int(n)).astype(np.int32) for n in lens]
    return shape, W, [prompts[int(np.argmin(lens))]], 64


def _fp8():
    # the block-FP8 test model (d 256, GQA 4/2, hd 64): W8A8 linear layers and the FP8 KV round trip
    shape = DecoderShape(2, 256, 4, 2, 64, 512, 1024)
    W = omodel.fp8_weights(omodel.weights_to_f32(make_decoder_weights(shape, seed=51, w_std=0.05)))
    P = make_prompts(5, 10, 150, shape.vocab, seed=52)
    return shape, W, P, 40


CASES = {
    "small": (_small, parity.E2E_MAX_SMALL, parity.E2E_MEAN_SMALL, ("fp64", "bf16p", "both")),
    "small_gqa": (_small_gqa, parity.E2E_MAX_SMALL, parity.E2E_MEAN_SMALL, ("fp64", "bf16p", "both")),
    "dense_decoder": (_dense, parity.E2E_MAX, parity.E2E_MEAN, ("fp64", "bf16p", "both")),
    "long_context": (_long, parity.E2E_MAX_LONG, parity.E2E_MEAN_LONG, ("bf16p", "both")),
    "fp8": (_fp8, parity.E2E_MAX_FP8, parity.E2E_MEAN_FP8, ("fp64", "bf16p", "both")),
}


@pytest.mark.parametrize("name", list(CASES))
def test_free_running_bound_sits_on_the_measured_floor(name):
    build, bound_max, bound_mean, variants = CASES[name]
    shape, W, prompts, n_gen = build()
    rng = np.random.default_rng(7)
    gens = [rng.integers(0, shape.vocab, n_gen) for _ in prompts]
    res = floors(W, shape, prompts, gens, variants)
    f_max = max(v[0] for v in res.values())
    f_mean = max(v[1] for v in res.values())
    print(name, {k: tuple(f"{x:.2e}" for x in v) for k, v in res.items()})
    assert f_max <= bound_max <= SLACK * f_max, (name, f_max, bound_max)
    assert f_mean <= bound_mean <= SLACK * f_mean, (name, f_mean, bound_mean)


def test_bf16_ulp_is_one_step_of_the_bf16_bit_pattern():
    """The ulp that bf16_close scales by is the distance to the next bf16 value
    (the pattern plus one), at the bottom and top of binades, subnormals and 0."""
    import torch

    from tests.gpu_util import bf16_ulp
    xs = np.array([1.0, 1.5, 1.9921875, 2.0, 3.0, 0.75, 1e-3, 3.0e38, 2.0 ** -126, 2.0 ** -130, 0.0, -1.0, -2.5,
                   2.0 ** -126 * 1.5], np.float32)
    t = torch.from_numpy(xs).to(torch.bfloat16).abs()
    step = (t.view(torch.int16).int() + 1).to(torch.int16).view(torch.bfloat16).float() - t.float()
    assert np.array_equal(step.numpy().astype(np.float64), bf16_ulp(t.float().numpy()))
