"""Pins for the CPU oracle: each test ties a part of the oracle to something
other than itself -- the OCP FP8 definition, torch's own casts, closed forms,
brute force in float64, hand-derived values, and the layer's invariants.
These run without a GPU."""
import json
import math
import os

import numpy as np
import pytest
import torch

from ffn_side_attention_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------- formats
def test_e4m3_decode_matches_torch_all_codes(orc):
    codes = np.arange(256, dtype=np.uint8)
    ours = orc.e4m3_decode(codes)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    # sign of zero
    assert math.copysign(1, ours[0x80]) == -1.0


def test_e4m3_golden_points(orc):
    with open(os.path.join(GOLDEN, "e4m3_ocp_points.txt")) as f:
        rows = [ln.split()[:2] for ln in f if ln.strip() and not ln.startswith("#")]
    for code_s, val_s in rows:
        code = int(code_s, 16)
        got = float(orc.e4m3_decode([code])[0])
        if val_s == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val_s) and math.copysign(1, got) == math.copysign(1, float(val_s))
            assert int(orc.e4m3_encode([float(val_s)])[0]) == code


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(0)
    mags = np.concatenate([
        rng.uniform(0, 2 ** -6, 2000),            # subnormal range
        np.exp2(rng.uniform(-9, 8.8, 4000)),      # normals
        rng.uniform(0, 448, 2000),
    ]).astype(np.float32)
    vals = mags * np.where(rng.random(mags.shape) < 0.5, -1, 1).astype(np.float32)
    # exact midpoints between neighbouring codes: ties go to the even code
    pos = orc.e4m3_decode(np.arange(0, 0x7f, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids, pos.astype(np.float32)])
    ours = orc.e4m3_encode(vals)
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_e4m3_encode_saturates(orc):
    for v in [448.0, 449.0, 463.9, 464.0, 465.0, 1e6, float("inf")]:
        assert int(orc.e4m3_encode([v])[0]) == 0x7E
        assert int(orc.e4m3_encode([-v])[0]) == 0xFE
    assert int(orc.e4m3_encode([float("nan")])[0]) == 0x7F


def test_bf16_round_matches_torch(orc):
    rng = np.random.default_rng(1)
    x = rng.standard_normal(20000).astype(np.float32) * np.exp2(rng.integers(-30, 30, 20000)).astype(np.float32)
    # exact ties: bf16 value + half an ulp
    base = torch.from_numpy(x[:2000]).bfloat16().float().numpy()
    ties = (base.view(np.uint32) | np.uint32(0x8000)).view(np.float32)
    x = np.concatenate([x, ties])
    ours = orc.bf16_bits(x)
    ref = torch.from_numpy(x).bfloat16().view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_quantize_rows_rule(orc):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((5, 384)).astype(np.float32)
    x[1, 128:256] = 0.0                                   # an all-zero block
    x[2] *= 1e-3
    q, s = orc.quantize_rows(x)
    for r in range(5):
        for b in range(3):
            blk = x[r, 128 * b:128 * (b + 1)]
            amax = np.abs(blk).max()
            if amax == 0:
                assert s[r, b] == 1.0 and not q[r, 128 * b:128 * (b + 1)].any()
                continue
            assert s[r, b] == np.float32(amax) / np.float32(448.0)
            # library routine: torch's e4m3 cast of x/scale (fp32 division)
            ref = torch.from_numpy((blk / s[r, b]).astype(np.float32)).to(torch.float8_e4m3fn)
            assert np.array_equal(q[r, 128 * b:128 * (b + 1)], ref.view(torch.uint8).numpy())
            # the element holding amax encodes to +-448
            i = int(np.argmax(np.abs(blk)))
            assert q[r, 128 * b + i] & 0x7F == 0x7E
            # dequantised error within half an e4m3 ulp (relative 2^-4) plus the subnormal step
            deq = orc.e4m3_decode(q[r, 128 * b:128 * (b + 1)]) * s[r, b]
            assert np.all(np.abs(deq - blk) <= np.abs(blk) * 2.0 ** -4 + s[r, b] * 2.0 ** -10 + 1e-30)


# --------------------------------------------------------------------- router
def _bf16_vals(rng, shape, scale=1.0):
    return torch.from_numpy((rng.standard_normal(shape) * scale).astype(np.float32)).bfloat16().float().numpy()


@pytest.mark.parametrize("H", [8, 128, 264, 4096, 7168])
def test_canonical_dot_error_bound(orc, H):
    """|s - exact| <= gamma_n * sum|x w| for the lane chains (n = H/32 + 8
    steps, fma rounding once per step) plus the 5 folding levels."""
    rng = np.random.default_rng(H)
    for _ in range(20):
        x = _bf16_vals(rng, H)
        w = _bf16_vals(rng, H, 1 / math.sqrt(H))
        s = float(orc.canonical_dot(x, w))
        exact = math.fsum((x.astype(np.float64) * w.astype(np.float64)).tolist())
        n = H // 32 + 8 + 5
        u = 2.0 ** -24
        bound = (n * u / (1 - n * u)) * float(np.sum(np.abs(x.astype(np.float64) * w)))
        assert abs(s - exact) <= bound


def test_canonical_dot_one_hot_every_channel(orc):
    """x = e_h picks w[h] exactly: catches a dropped channel or a shifted index."""
    H = 264
    w = np.arange(1, H + 1, dtype=np.float32)
    for h in range(H):
        x = np.zeros(H, np.float32)
        x[h] = 1.0
        assert float(orc.canonical_dot(x, w)) == float(h + 1)


def test_canonical_dot_fold_order(orc):
    """Hand-derived value that only the canonical fold gives.  Lane 0 holds 1
    (channel 0), lanes 8 and 24 hold 2^-24 (chunks 8 and 24 = channels 64 and
    192).  Fold: level 16 gives p0 = 1 and p8 = 2^-24 + 2^-24 = 2^-23, level 8
    gives 1 + 2^-23 exactly.  A left-to-right sum would round 1 + 2^-24 to 1
    twice and give 1."""
    H = 256
    x = np.zeros(H, np.float32)
    w = np.ones(H, np.float32)
    x[0] = 1.0
    x[64] = 2.0 ** -24
    x[192] = 2.0 ** -24
    assert float(orc.canonical_dot(x, w)) == 1.0 + 2.0 ** -23
    seq = np.float32(0)
    for v in x:
        seq = np.float32(seq + v)
    assert float(seq) == 1.0


def test_router_zero_weights_tie_break(orc):
    """W_r = 0: all logits tie, so the top-k are experts 0..k-1 in that order
    with weight 1/k each."""
    T, H, E, k = 7, 64, 16, 5
    x = _bf16_vals(np.random.default_rng(3), (T, H))
    logits = orc.router_logits(x, np.zeros((H, E), np.float32), "fp32")
    idx, w = orc.topk(logits, k)
    assert (idx == np.arange(k)).all()
    assert np.allclose(w, 1.0 / k, rtol=0, atol=1e-7)


def test_router_planted_logits(orc):
    """One-hot router columns: logit e = x[e] * c_e (exact), so the top-k is
    known by construction; ties at equal planted values go to the lower id."""
    T, H, E, k = 4, 32, 8, 3
    c = np.array([1, 2, 3, 4, 5, 6, 7, 8], np.float32)
    Wr = np.zeros((H, E), np.float32)
    for e in range(E):
        Wr[e, e] = c[e]
    x = np.zeros((T, H), np.float32)
    x[0, :E] = [1, 1, 1, 1, 1, 1, 1, 1]           # logits = c -> 7, 6, 5
    x[1, :E] = [8, 4, 0, 2, 1.6, 0, 0, 0]         # logits 8, 8, 0, 8, 8 -> 0, 1, 3
    x[2, :E] = [-1, -1, -1, -1, -1, -1, -1, -1]   # -> 0, 1, 2
    x[3, :E] = [0, 0, 0, 0, 0, 0, 0, 0.125]       # logit 1 at 7, zeros -> 7, 0, 1
    idx, w = orc.topk(orc.router_logits(x, Wr, "fp32"), k)
    assert idx.tolist() == [[7, 6, 5], [0, 1, 3], [0, 1, 2], [7, 0, 1]]
    assert np.allclose(w[1], 1 / 3, atol=1e-7)


def test_router_bias_added_last_hand_value(orc):
    """The bias enters as one fp32 addition after the fold ("MoE 大规模分布式推理工程实战",
    section 4.1: logits of the linear gate, then + the bias, then top-k).  Hand value:
    lane 0 holds 1 (channel 0), lanes 8 and 24 hold 2^-24 (channels 64 and 192); the fold
    gives s = 1 + 2^-23 (level 16: 2^-24 + 2^-24 = 2^-23 exactly; level 8: 1 + 2^-23).
    With bias 2^-24, s + b = 1 + 3*2^-24 lies half-way between 1 + 2^-23 (odd mantissa) and
    1 + 2^-22 (even), so the logit is 1 + 2^-22.  Each wrong placement gives another value:
    no bias 1 + 2^-23; bias subtracted: 1 + 2^-24 ties to 1; bias added to lane 0 before
    the fold: 1 + 2^-24 ties to 1 there, and the fold then gives 1 + 2^-23."""
    H = 256
    x = np.zeros((1, H), np.float32)
    x[0, 0], x[0, 64], x[0, 192] = 1.0, 2.0 ** -24, 2.0 ** -24
    w = np.ones((H, 1), np.float32)
    got = float(orc.router_logits(x, w, "fp32", np.array([2.0 ** -24], np.float32))[0, 0])
    assert got == 1.0 + 2.0 ** -22
    assert float(orc.router_logits(x, w, "fp32")[0, 0]) == 1.0 + 2.0 ** -23
    # bf16 activations take the same route: all values above are bf16-exact
    xb = orc.bf16_bits(x)
    wb = orc.bf16_bits(w)
    assert float(orc.router_logits(xb, wb, "bf16", np.array([2.0 ** -24], np.float32))[0, 0]) == 1.0 + 2.0 ** -22


def test_router_bias_reorders_planted_topk(orc):
    """One-hot router columns plant logits c_e * x[e] (exact); a bias then moves experts
    in and out of the top-k.  Expected sets by hand: logits 1..8 plus bias
    (+10, 0, 0, 0, 0, -0.5, 0, -10) = (11, 2, 3, 4, 5, 5.5, 7, -2) -> top-3 = 0, 6, 5;
    without the bias (or with it subtracted) the top-3 would be 7, 6, 5.  A bias that
    makes two logits equal sends the tie to the lower id: (1..8) + (0, 0, 0, 0, 0, 0, 1, 0)
    = (..., 6, 8, 8) -> 6, 7, 5.  Weights are the softmax of the biased selected logits."""
    H, E, k = 16, 8, 3
    Wr = np.zeros((H, E), np.float32)
    for e in range(E):
        Wr[e, e] = float(e + 1)
    x = np.zeros((2, H), np.float32)
    x[:, :E] = 1.0
    b1 = np.array([10, 0, 0, 0, 0, -0.5, 0, -10], np.float32)
    idx, w = orc.topk(orc.router_logits(x, Wr, "fp32", b1), k)
    assert idx.tolist() == [[0, 6, 5]] * 2
    sel = np.array([11.0, 7.0, 5.5])
    p = np.exp(sel - sel.max())
    assert np.allclose(w[0], p / p.sum(), rtol=1e-6, atol=0)
    b2 = np.array([0, 0, 0, 0, 0, 0, 1, 0], np.float32)
    idx2, w2 = orc.topk(orc.router_logits(x, Wr, "fp32", b2), k)
    assert idx2.tolist() == [[6, 7, 5]] * 2
    p2 = np.exp(np.array([8.0, 8.0, 6.0]) - 8.0)
    assert np.allclose(w2[0], p2 / p2.sum(), rtol=1e-6, atol=0)


def test_router_bias_k_equals_E_is_softmax_of_biased_logits(orc):
    """k = E with a Zipf(1.2) log-bias: the weights are the full softmax of (x W + b),
    computed here in float64 from the matrix product (closed form), and the slots are the
    experts in descending biased-logit order.  The bias is ~ -6.7 .. 0, far above the
    canonical sum's rounding, so dropping or flipping it fails by orders of magnitude."""
    from scipy.special import softmax

    T, H, E = 40, 256, 16
    rng = np.random.default_rng(21)
    x = _bf16_vals(rng, (T, H))
    Wr = _bf16_vals(rng, (H, E), 1 / math.sqrt(H))
    b = synth.zipf_bias(E, 1.2).numpy()
    idx, w = orc.topk(orc.router_logits(orc.bf16_bits(x), orc.bf16_bits(Wr), "bf16", b), E)
    z = x.astype(np.float64) @ Wr.astype(np.float64) + b.astype(np.float64)
    p = softmax(z, axis=1)
    for t in range(T):
        assert idx[t].tolist() == sorted(range(E), key=lambda e: (-z[t, e], e))
        assert np.allclose(w[t], p[t, idx[t]], rtol=1e-5, atol=1e-7)


def test_topk_brute_force(orc):
    rng = np.random.default_rng(4)
    T, E, k = 300, 40, 6
    logits = rng.standard_normal((T, E)).astype(np.float32)
    logits[:50, :] = np.round(logits[:50, :])  # many exact ties
    idx, w = orc.topk(logits, k)
    for t in range(T):
        order = sorted(range(E), key=lambda e: (-float(logits[t, e]), e))[:k]
        assert idx[t].tolist() == order
        sel = logits[t, order].astype(np.float64)
        p = np.exp(sel - sel.max())
        assert np.allclose(w[t], p / p.sum(), rtol=1e-6, atol=0)
        assert abs(float(w[t].astype(np.float64).sum()) - 1.0) < 1e-6


def test_topk_k_equals_E_is_full_softmax(orc):
    from scipy.special import softmax

    rng = np.random.default_rng(5)
    logits = rng.standard_normal((50, 12)).astype(np.float32)
    idx, w = orc.topk(logits, 12)
    full = softmax(logits.astype(np.float64), axis=1)
    for t in range(50):
        assert np.allclose(w[t], full[t, idx[t]], rtol=1e-6)


def test_routing_tables_invariants(orc):
    rng = np.random.default_rng(6)
    T, E, k = 333, 24, 4
    idx = np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)
    counts, offsets, perm, pos = orc.routing_tables(idx, E)
    assert counts.sum() == T * k
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts))
    assert sorted(pos.tolist()) == list(range(T * k))  # bijection onto packed rows
    for t in range(T):
        for j in range(k):
            r = pos[t * k + j]
            e = idx[t, j]
            assert perm[r] == t and offsets[e] <= r < offsets[e + 1]
    for e in range(E):
        seg = perm[offsets[e]:offsets[e + 1]]
        assert np.all(np.diff(seg) > 0)  # ascending token order within an expert
        assert np.array_equal(seg, np.nonzero((idx == e).any(axis=1))[0])


# --------------------------------------------------------------------- full layer
def _np_swiglu(a, wg, wu, wd):
    g = a @ wg
    return ((g / (1 + np.exp(-g))) * (a @ wu)) @ wd


def _tiny(dtype="fp32", E=8, k=2, S=0, H=128, I=256, B=32, M=2):
    return synth.LayerConfig("t", H=H, I=I, E=E, k=k, S=S, dtype=dtype, B=B, M=M)


def _cfgd(c):
    return dict(H=c.H, I=c.I, E=c.E, k=c.k, S=c.S, dtype=c.dtype)


def test_golden_hand_example(orc):
    with open(os.path.join(GOLDEN, "tiny_hand_moe.json")) as f:
        g = json.load(f)
    H, I, E = g["H"], g["I"], g["E"]
    wr = np.zeros((H, E), np.float32)
    wr[0, :] = g["router_col"]
    wg = np.zeros((E, H, I), np.float32)
    wu = np.zeros((E, H, I), np.float32)
    wd = np.zeros((E, I, H), np.float32)
    for e in range(E):
        wg[e, 0, 0] = g["gate00"][e]
        wu[e, 0, 0] = g["up00"][e]
        wd[e, 0, :] = g["down_row0"][e]
    x = np.array([g["x"]], np.float32)
    weights = dict(w_router=wr, w_gate=wg, w_up=wu, w_down=wd)
    r1 = orc.moe_forward(dict(H=H, I=I, E=E, k=1, S=0, dtype="fp32"), [x], weights)
    assert r1["out"][0].tolist() == g["out_k1"] and r1["idx"].tolist() == [[0]]
    r2 = orc.moe_forward(dict(H=H, I=I, E=E, k=2, S=0, dtype="fp32"), [x], weights)
    assert np.allclose(r2["w"][0], g["w_k2"], rtol=1e-7)
    assert np.allclose(r2["out"][0], g["out_k2"], rtol=1e-6)


def test_identical_experts_equal_dense_swiglu(orc):
    c = _tiny()
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    for key in ("w_gate", "w_up", "w_down"):
        w[key] = np.repeat(w[key][:1], c.E, axis=0)
    r = orc.moe_forward(_cfgd(c), src, w)
    x = np.concatenate(src).astype(np.float64)
    ref = _np_swiglu(x, w["w_gate"][0].astype(np.float64), w["w_up"][0].astype(np.float64),
                     w["w_down"][0].astype(np.float64))
    err = np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref)
    assert err < 1e-6


def test_zero_input_gives_zero(orc):
    c = _tiny()
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), [np.zeros((5, c.H), np.float32)], w)
    assert not r["out"].any()


def test_single_expert_is_textbook_swiglu(orc):
    c = _tiny(E=1, k=1)
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), src, w)
    assert np.allclose(r["w"], 1.0)
    x = np.concatenate(src).astype(np.float64)
    ref = _np_swiglu(x, w["w_gate"][0].astype(np.float64), w["w_up"][0].astype(np.float64),
                     w["w_down"][0].astype(np.float64))
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-6


def test_k_equals_E_is_full_softmax_mixture(orc):
    from scipy.special import softmax

    c = _tiny(E=4, k=4)
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), src, w)
    x = np.concatenate(src).astype(np.float64)
    p = softmax(x @ w["w_router"].astype(np.float64), axis=1)
    ref = sum(p[:, e:e + 1] * _np_swiglu(x, w["w_gate"][e].astype(np.float64), w["w_up"][e].astype(np.float64),
                                         w["w_down"][e].astype(np.float64)) for e in range(c.E))
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-5


def test_k_equals_E_with_bias_is_biased_softmax_mixture(orc):
    """The layer passes the router bias through to routing: with k = E and a bias, the
    output is the mixture weighted by softmax(x W_r + b) (closed form in float64)."""
    from scipy.special import softmax

    c = _tiny(E=4, k=4)
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    w["router_bias"] = np.array([1.5, -2.0, 0.25, 0.0], np.float32)
    r = orc.moe_forward(_cfgd(c), src, w)
    x = np.concatenate(src).astype(np.float64)
    p = softmax(x @ w["w_router"].astype(np.float64) + w["router_bias"].astype(np.float64), axis=1)
    ref = sum(p[:, e:e + 1] * _np_swiglu(x, w["w_gate"][e].astype(np.float64), w["w_up"][e].astype(np.float64),
                                         w["w_down"][e].astype(np.float64)) for e in range(c.E))
    assert np.linalg.norm(r["out"] - ref) / np.linalg.norm(ref) < 1e-5
    no_bias = orc.moe_forward(_cfgd(c), src, {k_: v for k_, v in w.items() if k_ != "router_bias"})
    assert np.linalg.norm(no_bias["out"] - ref) / np.linalg.norm(ref) > 1e-2


def test_shared_expert_adds_unweighted(orc):
    c = _tiny(S=1)
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), src, w)
    r0 = orc.moe_forward(_cfgd(_tiny(S=0)), src, {k: v for k, v in w.items() if not k.startswith("sh_")})
    x = np.concatenate(src).astype(np.float64)
    sh = _np_swiglu(x, w["sh_gate"].astype(np.float64), w["sh_up"].astype(np.float64), w["sh_down"].astype(np.float64))
    assert np.linalg.norm(r["out"] - r0["out"] - sh) / np.linalg.norm(sh) < 1e-5


def test_token_order_and_buffer_split_invariance(orc):
    """Each token's output depends only on that token: permuting tokens
    permutes outputs bit for bit, and regrouping rows into other buffers
    (including empty ones) changes nothing."""
    c = _tiny()
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    base = orc.moe_forward(_cfgd(c), src, w)
    x = np.concatenate(src)
    p = np.random.default_rng(7).permutation(x.shape[0])
    rp = orc.moe_forward(_cfgd(c), [x[p]], w)
    assert np.array_equal(rp["out"], base["out"][p]) and np.array_equal(rp["idx"], base["idx"][p])
    parts = [x[:5], x[5:5], x[5:40], x[40:]]
    rs = orc.moe_forward(_cfgd(c), parts, w)
    assert np.array_equal(rs["out"], base["out"])
    sub = orc.moe_forward(_cfgd(c), src, w, tokens=[63, 0, 17])
    assert np.array_equal(sub["out"], base["out"][[63, 0, 17]])


def test_thread_count_does_not_change_results(orc):
    """The bench times the oracle on one core and on all of them; each parallel loop
    writes its own tokens' results, so the thread count changes nothing."""
    c = _tiny(S=1)
    src = [s.numpy() for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    n = orc.num_threads()
    try:
        orc.set_num_threads(1)
        one = orc.moe_forward(_cfgd(c), src, w)
    finally:
        orc.set_num_threads(n)
    many = orc.moe_forward(_cfgd(c), src, w)
    for key in ("out", "idx", "w", "logits"):
        assert np.array_equal(one[key], many[key]), key
    assert one["fma"] == many["fma"]


def test_flop_count(orc):
    for S in (0, 1):
        c = _tiny(S=S)
        src = [s.numpy() for s in synth.make_sources(c)]
        w = synth.weights_numpy(synth.make_weights(c))
        r = orc.moe_forward(_cfgd(c), src, w)
        assert 2 * r["fma"] == 6 * c.T * (c.k + S) * c.H * c.I


def test_empty_batch(orc):
    c = _tiny()
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), [np.zeros((0, c.H), np.float32)] * 3, w)
    assert r["out"].shape == (0, c.H)


def test_bf16_layer_matches_float64_reference(orc):
    """bf16 layer: operands are exact bf16 values, so a float64 reference that
    rounds h to bf16 with torch's cast reproduces the oracle to ~1e-6."""
    c = _tiny(dtype="bf16", H=256, I=256, E=4, k=2)
    src = [synth.to_numpy_bits(s) for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), src, w)
    f = orc.bf16_to_f32
    x = np.concatenate([f(s) for s in src]).astype(np.float64)
    out = np.zeros_like(x)
    for t in range(x.shape[0]):
        for j in range(c.k):
            e = r["idx"][t, j]
            g = x[t] @ f(w["w_gate"][e]).astype(np.float64)
            u = x[t] @ f(w["w_up"][e]).astype(np.float64)
            h = torch.from_numpy((g / (1 + np.exp(-g)) * u).astype(np.float32)).bfloat16().double().numpy()
            out[t] += float(r["w"][t, j]) * (h @ f(w["w_down"][e]).astype(np.float64))
    got = f(r["out"]).astype(np.float64)
    assert np.linalg.norm(got - out) / np.linalg.norm(out) < 4e-3  # output rounded to bf16 once
    assert np.abs(got - out).max() <= np.abs(out).max() * 2 ** -8


def test_fp8_layer_matches_float64_reference(orc):
    """fp8 layer: activations quantised per token per 128 channels with torch's
    e4m3 cast, weights dequantised block-wise -- float64 reference agrees."""
    c = _tiny(dtype="fp8", H=256, I=256, E=4, k=2, S=1)
    src = [synth.to_numpy_bits(s) for s in synth.make_sources(c)]
    w = synth.weights_numpy(synth.make_weights(c))
    r = orc.moe_forward(_cfgd(c), src, w)
    f = orc.bf16_to_f32

    def deq_w(q, s):
        v = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).double().numpy()
        return v * np.kron(s.astype(np.float64), np.ones((128, 128)))

    def qrow(v):
        v = v.astype(np.float32)
        out = np.zeros(v.shape, np.float64)
        for b in range(0, v.shape[0], 128):
            blk = v[b:b + 128]
            amax = np.abs(blk).max()
            if amax == 0:
                continue
            sc = np.float32(amax) / np.float32(448)
            out[b:b + 128] = torch.from_numpy(blk / sc).to(torch.float8_e4m3fn).double().numpy() * float(sc)
        return out

    x = np.concatenate([f(s) for s in src])
    ref = np.zeros(x.shape, np.float64)
    for t in range(x.shape[0]):
        a = qrow(x[t])
        experts = [(r["idx"][t, j], float(r["w"][t, j]), "") for j in range(c.k)] + [(0, 1.0, "sh_")]
        for e, wj, p in experts:
            if p:
                wg, wu, wd = (deq_w(w["sh_gate"], w["sh_s_gate"]), deq_w(w["sh_up"], w["sh_s_up"]),
                              deq_w(w["sh_down"], w["sh_s_down"]))
            else:
                wg, wu, wd = (deq_w(w["w_gate"][e], w["s_gate"][e]), deq_w(w["w_up"][e], w["s_up"][e]),
                              deq_w(w["w_down"][e], w["s_down"][e]))
            g = a @ wg
            h = qrow((g / (1 + np.exp(-g)) * (a @ wu)).astype(np.float32))
            ref[t] += wj * (h @ wd)
    got = f(r["out"]).astype(np.float64)
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 4e-3


@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp8"])
def test_expert_hidden_matches_float64_swiglu(orc, dtype):
    """The hidden-row export (silu(a Wg) * (a Wu) rounded once to fp32, per (token,
    expert)) against a float64 numpy evaluation: a = the token in the layer's operand
    format (fp32 / bf16 values / torch's e4m3 cast per 128 channels), weights dequantised
    block-wise for fp8.  The two sums differ only in float64 rounding order, so after the
    fp32 rounding they agree to one fp32 ulp.  The shared expert is selected by id -1."""
    c = _tiny(dtype=dtype, H=256, I=256, E=4, k=2, S=1)
    src = synth.make_sources(c)
    x = np.concatenate([synth.to_numpy_bits(s) for s in src])[:24]
    w = synth.weights_numpy(synth.make_weights(c))
    experts = np.array([t % c.E for t in range(23)] + [-1], np.int32)
    got = orc.expert_hidden(_cfgd(c), w, x, experts)
    xf = x.astype(np.float32) if dtype == "fp32" else orc.bf16_to_f32(x)

    def wmat(key, e):
        if dtype == "fp32":
            return w[key][e].astype(np.float64) if e >= 0 else w["sh_" + key[2:]].astype(np.float64)
        q = w[key][e] if e >= 0 else w["sh_" + key[2:]]
        if dtype == "bf16":
            return orc.bf16_to_f32(q).astype(np.float64)
        s = w["s_" + key[2:]][e] if e >= 0 else w["sh_s_" + key[2:]]
        v = torch.from_numpy(q.copy()).view(torch.float8_e4m3fn).double().numpy()
        return v * np.kron(s.astype(np.float64), np.ones((128, 128)))

    def operand(row):
        if dtype != "fp8":
            return row.astype(np.float64)
        out = np.zeros(row.shape, np.float64)
        for b in range(0, row.shape[0], 128):
            blk = row[b:b + 128].astype(np.float32)
            sc = np.float32(np.abs(blk).max()) / np.float32(448)
            out[b:b + 128] = torch.from_numpy(blk / sc).to(torch.float8_e4m3fn).double().numpy() * float(sc)
        return out

    for i, e in enumerate(experts):
        a = operand(xf[i])
        g = a @ wmat("w_gate", e)
        ref = (g / (1 + np.exp(-g)) * (a @ wmat("w_up", e))).astype(np.float32)
        ulp = np.spacing(np.abs(ref)).astype(np.float64)
        assert np.all(np.abs(got[i].astype(np.float64) - ref) <= ulp), f"row {i} expert {e}"
    with pytest.raises(ValueError):
        orc.expert_hidden(_cfgd(c), w, x[:1], np.array([c.E], np.int32))
