"""The synthetic input recipe: seeded and reproducible, the stated distributions,
the fp8 block format, and the Zipf(1.2) router bias over a seeded expert
permutation (so softmax weights are scaled by a Zipf pmf over expert ranks)."""
import math

import numpy as np
import torch

from ffn_side_attention_gb300 import synth


def _small(dtype, **kw):
    base = dict(H=256, I=256, E=16, k=4, S=1, dtype=dtype, B=0, M=0)
    base.update(kw)
    return synth.LayerConfig("small", **base)


def test_sources_are_seeded_split_and_normal():
    c = _small("bf16")
    a = synth.make_sources(c, counts=[300, 0, 212], seed=3)
    b = synth.make_sources(c, counts=[512], seed=3)
    assert [x.shape[0] for x in a] == [300, 0, 212] and all(x.dtype == torch.bfloat16 for x in a)
    assert torch.equal(torch.cat(a), b[0])  # the split into buffers does not change the rows
    assert not torch.equal(b[0], synth.make_sources(c, counts=[512], seed=4)[0])
    x = b[0].float()
    assert abs(x.mean().item()) < 0.02 and abs(x.std().item() - 1.0) < 0.02


def test_weights_follow_fan_in():
    c = _small("fp32", H=512, I=384)
    w = synth.make_weights(c)
    assert abs(w["w_router"].std().item() * math.sqrt(512) - 1.0) < 0.05
    assert abs(w["w_gate"].std().item() * math.sqrt(512) - 1.0) < 0.02
    assert abs(w["w_down"].std().item() * math.sqrt(384) - 1.0) < 0.02
    w2 = synth.make_weights(c)
    assert all(torch.equal(w[k], w2[k]) for k in w)


def test_fp8_weights_are_block_quantised_codes_and_scales():
    c = _small("fp8", E=2, S=0)
    w = synth.make_weights(c)
    q = w["w_gate"][0].view(torch.float8_e4m3fn).float()      # [H, I] codes
    s = w["s_gate"][0]                                         # [H/128, I/128]
    assert q.shape == (256, 256) and s.shape == (2, 2)
    for i in range(2):
        for j in range(2):
            blk = q[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)]
            assert blk.abs().max().item() == 448.0             # scale = block amax / 448
    # the dequantised values are the fp32 master weights up to e4m3 rounding
    g = synth._gen("cpu", 0, synth.SUB_EXPERT0 + 0)
    master = torch.randn(256, 256, generator=g) / 16.0
    deq = q * s.repeat_interleave(128, 0).repeat_interleave(128, 1)
    rel = (deq - master).abs() / master.abs().clamp_min(1e-3)
    assert np.percentile(rel.numpy(), 99) < 2 ** -3


def test_zipf_bias_is_log_pmf_over_a_permutation():
    b = synth.zipf_bias(256, 1.2, seed=0).double()
    ranks = torch.round(torch.exp(-b / 1.2) - 1.0).long()
    assert sorted(ranks.tolist()) == list(range(256))          # a permutation of 0..E-1
    assert torch.allclose(b, -1.2 * torch.log(ranks.double() + 1.0), atol=1e-6)
    assert ranks.tolist() != list(range(256))                  # seeded shuffle, not the identity
    # exp(bias) ratios are Zipf(1.2) pmf ratios between ranks
    e0, e9 = int((ranks == 0).nonzero()), int((ranks == 9).nonzero())
    assert abs(math.exp(b[e9] - b[e0]) - 10.0 ** -1.2) < 1e-6
    assert torch.equal(synth.zipf_bias(256, 1.2, seed=0), synth.zipf_bias(256, 1.2, seed=0))
