"""Weights updated in place between RL steps.

"vLLM Achieves Bitwise-Consistent RL Training ..." §4.6: a captured CUDA graph
keeps the addresses of the buffers it was captured on, so the trainer copies new
weights into the same buffers, and the comparison has to hold again after the
update.  Here one Episode (static buffers, one decode graph captured on the first
run) runs an RL step, the weights are overwritten in place (for the block-FP8
model the FP8 copies are re-made from the new bf16 masters by `requantize()`,
the deployment rule), and the next step must again give rollout == recompute
bitwise, and must equal, bit for bit, a fresh decoder built on the new weights
and run eagerly (so the replayed graph really read the new values).
"""
import numpy as np
import pytest
import torch

import invariant_forward_policy_gb300 as bi
from invariant_forward_policy_gb300.decoder import Decoder, Episode
from synthetic import DecoderShape, make_decoder_weights, make_prompts
from tests.gpu_util import same_bits

pytestmark = pytest.mark.gpu


def _copy_weights_in_place(dec, wb):
    """Overwrite every weight buffer of `dec` with the bf16 bit arrays of `wb` (same shapes)."""
    def put(dst, bits):
        src = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)
        assert dst.shape == src.shape
        dst.copy_(src.to(dst.device))
    for k in ("embed", "final_norm", "lm_head"):
        put(dec.w[k], wb[k])
    for lw, lb in zip(dec.layers, wb["layers"]):
        for k, bits in lb.items():
            put(lw[k], bits)
    if dec.fp8:
        dec.requantize()


@pytest.mark.parametrize("fp8", [False, True])
def test_weights_updated_in_place_keep_rollout_equal_to_recompute(fp8):
    shape = DecoderShape(2, 128, 4, 2, 64, 256, 512) if not fp8 else DecoderShape(2, 256, 4, 2, 64, 512, 1024)
    wa = make_decoder_weights(shape, seed=61, w_std=0.05)
    wb = make_decoder_weights(shape, seed=62, w_std=0.05)
    prompts = make_prompts(4, 20, 90, shape.vocab, seed=63)
    n_gen = 24
    pd = torch.from_numpy(np.concatenate(prompts).astype(np.int32)).cuda()
    dec = Decoder(shape, wa, max_pos=512, fp8=fp8)
    ep = Episode(dec, [len(p) for p in prompts], n_gen)
    ids_a, lp_a, rec_a = (t.clone() for t in ep.run(pd))          # first step captures the decode graph
    assert same_bits(lp_a, rec_a)
    _copy_weights_in_place(dec, wb)
    ids_b, lp_b, rec_b = (t.clone() for t in ep.run(pd))          # the same graph, replayed on new weights
    torch.cuda.synchronize()
    assert same_bits(lp_b, rec_b)
    assert not same_bits(lp_a, lp_b)                              # the update reached the replayed kernels
    # a decoder built on the new weights from scratch, decoding eagerly, gives the same bits
    fresh = Decoder(shape, wb, max_pos=512, fp8=fp8)
    lens = [len(p) for p in prompts]
    mb = -(-(max(lens) + n_gen) // 64)
    ids_f, lp_f = fresh.rollout(prompts, n_gen, fresh.alloc_cache(4 * mb), fresh.block_table(4, mb, seed=5),
                                use_graph=False)
    assert torch.equal(ids_f, ids_b) and same_bits(lp_f, lp_b)
    # and back: restoring the old weights in place restores the old step exactly
    _copy_weights_in_place(dec, wa)
    ids_r, lp_r, rec_r = ep.run(pd)
    torch.cuda.synchronize()
    assert torch.equal(ids_r, ids_a) and same_bits(lp_r, lp_a) and same_bits(rec_r, rec_a)
    assert bi.bi_device_status() == 0
