"""GPU parity of the expert-GEMM operands, code for code.

The packed token rows P (and, for the fp8 layer, their e4m3 codes and fp32 scales per
128 channels) must equal the oracle's quantisation of the same tokens bit for bit: both
sides quantise identical bf16 inputs by the same rule ("MoE系统与AFD架构概述", section
3.3, FP8 activations; per token per 128 channels, scale = amax / 448, nearest-even
e4m3, saturating).  The SwiGLU rows h are the product of an fp32 tensor-core GEMM on
the GPU and of float64 sums in the oracle, so their pre-rounding values differ by a few
fp32 ulps; a code may then differ by one step, and only where the oracle's value lies
on a rounding boundary of the two codes.  That is checked element by element."""
import numpy as np
import pytest
import torch

import oracle
from ffn_side_attention_gb300 import synth

from gpu_helpers import cfg_dict, make_layer

pytestmark = pytest.mark.gpu

# A code flip is accepted only where the oracle's value, in units of the block scale, is
# this close (relative) to the midpoint of the two codes: the GPU's fp32 h differs from
# the oracle's by ~1e-6 relative, far inside this.
MID_REL = 2.0 ** -12
SCALE_REL = 1e-4  # scales follow amax, which carries the same ~1e-6 relative difference


def _e4m3_values():
    v = oracle.e4m3_decode(np.arange(256, dtype=np.uint8))
    return v


def _adjacent_rank(values: np.ndarray):
    """Rank of each finite code's value among the distinct finite e4m3 values (+0 and -0
    share one rank): adjacent codes in value order differ by one rank."""
    finite = np.isfinite(values)
    uniq = np.unique(values[finite])
    rank = np.full(256, -10 ** 6, np.int64)
    rank[finite] = np.searchsorted(uniq, values[finite])
    return rank


def _forward(c, counts, weights=None, seed=0):
    T = sum(counts)
    srcs = synth.make_sources(c, "cuda", seed=seed, counts=counts)
    w = weights if weights is not None else synth.make_weights(c, "cuda", seed=seed)
    layer = make_layer(c, w, max_tokens=T, max_sources=max(len(counts), 1))
    layer.forward(srcs)
    torch.cuda.synchronize()
    layer.check()
    r = layer.routing(T)
    ops = layer.operands(T)
    torch.cuda.synchronize()
    x = torch.cat(srcs)
    return layer, w, x, r, ops


def _row_tokens_experts(c, r, T):
    """Token and expert (-1 = shared) of every packed row."""
    k = c.k
    perm = r["perm"].cpu().numpy()
    offsets = r["offsets"].cpu().numpy()
    experts = np.repeat(np.arange(c.E), np.diff(offsets))
    tokens = perm
    if c.S:
        tokens = np.concatenate([tokens, np.arange(T)])
        experts = np.concatenate([experts, np.full(T, -1)])
    assert tokens.shape[0] == T * (k + c.S)
    return tokens.astype(np.int64), experts.astype(np.int32)


def _check_fp8_codes(got_codes, got_scales, ref_vals, label):
    """got_codes [n, C] uint8 and got_scales [n, C/128] against the oracle's fp32 values
    ref_vals [n, C] quantised by oracle.quantize_rows.  Returns the fraction of codes
    that differ (each one a boundary case)."""
    ref_codes, ref_scales = oracle.quantize_rows(ref_vals)
    rel = np.abs(got_scales.astype(np.float64) / ref_scales.astype(np.float64) - 1.0)
    assert rel.max() <= SCALE_REL, f"{label}: scale differs by {rel.max():.2e} relative"
    diff = got_codes != ref_codes
    if not diff.any():
        return 0.0
    vals = _e4m3_values()
    rank = _adjacent_rank(vals)
    rr, cc = np.nonzero(diff)
    a, b = got_codes[rr, cc], ref_codes[rr, cc]
    assert np.all(np.abs(rank[a] - rank[b]) == 1), f"{label}: a code differs by more than one step"
    mid = (vals[a] + vals[b]) / 2
    y = ref_vals[rr, cc].astype(np.float64) / ref_scales[rr, cc // 128].astype(np.float64)
    off = np.abs(y - mid) / np.maximum(np.abs(mid), 2.0 ** -9)
    assert off.max() <= MID_REL, f"{label}: a code differs away from a rounding boundary ({off.max():.2e})"
    return float(diff.mean())


# bf16 h: G and U are fp32 tensor-core sums of H products on the GPU and float64 sums in
# the oracle, so where G is near zero silu(G) * U carries an absolute difference of the
# order of the fp32 accumulation error (~1e-5 here), which can exceed one bf16 step of a
# small value.  A value may differ from the oracle's rounding by one bf16 step anywhere,
# or by at most H_ABS in absolute terms.
H_ABS = 2.0 ** -14


def _check_bf16_rounding(got_bits, ref_vals, label):
    """bf16 h against the oracle's fp32 values: equal to their nearest-even rounding except
    (a) one bf16 step away, or (b) within H_ABS of the oracle's value.  Returns the
    fraction of values that differ from the oracle's rounding."""
    ref_bits = oracle.bf16_bits(ref_vals)
    diff = got_bits != ref_bits
    if not diff.any():
        return 0.0
    ga, rb = got_bits[diff].astype(np.int64), ref_bits[diff].astype(np.int64)

    def order(bits):  # bf16 patterns in value order (+0 and -0 share a key)
        return np.where(bits < 0x8000, bits, -(bits & 0x7FFF))

    one_step = np.abs(order(ga) - order(rb)) == 1
    got = oracle.bf16_to_f32(got_bits[diff]).astype(np.float64)
    near = np.abs(got - ref_vals[diff].astype(np.float64)) <= H_ABS
    bad = ~(one_step | near)
    assert not bad.any(), (f"{label}: {int(bad.sum())} bf16 values differ by more than one step and "
                           f"{H_ABS:g}; worst {np.abs(got - ref_vals[diff])[bad].max():.3e}")
    return float(diff.mean())


def _sample_rows(n_rows, n, seed=3):
    rng = np.random.default_rng(seed)
    pick = set(rng.choice(n_rows, min(n, n_rows), replace=False).tolist())
    pick |= {0, n_rows - 1}
    return np.array(sorted(pick), np.int64)


def _fp8_case(c, counts, n_h_rows, weights=None):
    T = sum(counts)
    layer, w, x, r, ops = _forward(c, counts, weights)
    tokens, experts = _row_tokens_experts(c, r, T)
    xb = synth.to_numpy_bits(x)  # bf16 bits [T, H]
    # P: the oracle quantises each token once; packed rows are copies of their token's row
    xq, xs = oracle.quantize_rows(oracle.bf16_to_f32(xb))
    P = ops["P"].cpu().numpy()
    Ps = ops["P_scale"].cpu().numpy().T  # [R, H/128]
    assert np.array_equal(P, xq[tokens]), "packed e4m3 codes differ from the oracle's"
    assert np.array_equal(Ps.view(np.uint32), xs[tokens].view(np.uint32)), "packed scales differ from the oracle's"
    # h: sampled packed rows, oracle hidden values quantised by the oracle's rule
    rows = _sample_rows(tokens.shape[0], n_h_rows)
    hf = oracle.expert_hidden(cfg_dict(c), synth.weights_numpy(w), xb[tokens[rows]], experts[rows])
    got = ops["h"].cpu().numpy()[rows]
    gs = ops["h_scale"].cpu().numpy().T[rows]
    frac = _check_fp8_codes(got, gs, hf, c.name)
    layer.close()
    return frac


def test_fp8_operands_small_ragged_with_shared_expert():
    c = synth.LayerConfig("small_fp8", H=512, I=384, E=16, k=4, S=1, dtype="fp8", B=0, M=0)
    frac = _fp8_case(c, [17, 0, 40], n_h_rows=10 ** 6)  # every packed row
    assert frac <= 1e-2


def test_fp8_operands_qwen3_full_size():
    """qwen3_fp8 at T = 4 x 395: all 12640 packed rows of P bit for bit; h on 256 sampled rows."""
    c = synth.CONFIGS["qwen3_fp8"]
    frac = _fp8_case(c, [c.B] * c.M, n_h_rows=256)
    print(f"qwen3_fp8 h codes differing: {frac:.2e}")
    assert frac <= 1e-2


@pytest.mark.parametrize("B", [64, 512])
def test_fp8_operands_dsv3_zipf(B):
    """DeepSeek-V3 shapes with the Zipf-biased router and the shared expert, T = 8 x B:
    every packed row of P bit for bit; h on sampled rows (shared-expert rows included)."""
    c = synth.CONFIGS["dsv3_fp8"].with_batch(B, 8)
    frac = _fp8_case(c, [c.B] * c.M, n_h_rows=192)
    print(f"dsv3_fp8 T={c.T} h codes differing: {frac:.2e}")
    assert frac <= 1e-2


def test_bf16_operands_qwen3():
    """bf16 layer: packed rows are bit copies of their tokens; h is the nearest-even bf16
    of the oracle's fp32 SwiGLU value up to boundary cases."""
    c = synth.CONFIGS["qwen3_bf16"].with_batch(395, 2)
    T = c.T
    layer, w, x, r, ops = _forward(c, [c.B] * c.M)
    tokens, experts = _row_tokens_experts(c, r, T)
    xb = synth.to_numpy_bits(x)
    P = ops["P"].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(P, xb[tokens]), "packed bf16 rows differ from their tokens"
    rows = _sample_rows(tokens.shape[0], 256)
    hf = oracle.expert_hidden(cfg_dict(c), synth.weights_numpy(w), xb[tokens[rows]], experts[rows])
    got = ops["h"].view(torch.int16).cpu().numpy().view(np.uint16)[rows]
    frac = _check_bf16_rounding(got, hf, c.name)
    print(f"qwen3_bf16 h values differing: {frac:.2e}")
    assert frac <= 1e-2
    layer.close()


def test_bf16_small_batch_writes_no_P_and_h_follows_the_oracle():
    """A bf16 forward of at most 8 tokens packs no rows (its gate/up GEMM copies the token
    rows from the sources): P is rejected, and h, computed from those rows, is still the
    nearest-even bf16 of the oracle's SwiGLU value up to boundary cases (qwen3 shapes, 6
    tokens)."""
    from ffn_side_attention_gb300 import afd

    c = synth.CONFIGS["qwen3_bf16"].with_batch(6, 1)
    T = c.T
    srcs = synth.make_sources(c, "cuda", counts=[T])
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=T, max_sources=1)
    layer.forward(srcs)
    torch.cuda.synchronize()
    layer.check()
    r = layer.routing(T)
    ops = layer.operands(T, with_P=False)
    torch.cuda.synchronize()
    with pytest.raises(afd.AfdError) as e:
        layer.operands(T)
    assert e.value.code == afd.AFD_EINVAL
    tokens, experts = _row_tokens_experts(c, r, T)
    xb = synth.to_numpy_bits(torch.cat(srcs))
    hf = oracle.expert_hidden(cfg_dict(c), synth.weights_numpy(w), xb[tokens], experts)
    got = ops["h"].view(torch.int16).cpu().numpy().view(np.uint16)
    frac = _check_bf16_rounding(got, hf, c.name)
    print(f"qwen3_bf16 T=6 h values differing: {frac:.2e}")
    assert frac <= 1e-2
    layer.close()


def test_operand_scales_rejected_for_bf16():
    from ffn_side_attention_gb300 import afd

    c = synth.LayerConfig("small_bf16", H=256, I=256, E=8, k=2, S=0, dtype="bf16", B=0, M=0)
    layer, w, x, r, ops = _forward(c, [9])  # above 8 tokens: P is written
    dummy = torch.empty(16, dtype=torch.float32, device="cuda")
    with pytest.raises(afd.AfdError) as e:
        afd.afd_ffn_debug_operands(layer.handle, None, None, dummy.data_ptr(), None, None)
    assert e.value.code == afd.AFD_EINVAL
    layer.close()
