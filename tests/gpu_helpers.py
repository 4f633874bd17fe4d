"""Shared helpers for the GPU parity tests: run the CUDA layer through the C
ABI, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from ffn_side_attention_gb300 import afd, synth

# Tolerances: bf16 per the layer's BF16 criterion, fp8 per its FP8 criterion;
# fp32 from the fp32 arithmetic (FMA chains of <= 8K terms, single-precision
# silu/exp): relative Frobenius 1e-5, max-abs 1e-4.
TOL = {
    "fp32": dict(rel=1e-5, abs=1e-4),
    "bf16": dict(rel=1e-2, abs=5e-2),
    "fp8": dict(rel=3e-2, abs=None),
}
# routing weights: fp32 expf/division vs the oracle's double softmax
W_ATOL = 2e-6


def cfg_dict(c: synth.LayerConfig) -> dict:
    return dict(H=c.H, I=c.I, E=c.E, k=c.k, S=c.S, dtype=c.dtype)


def make_layer(c: synth.LayerConfig, w: dict, max_tokens: int, max_sources: int = 16) -> afd.MoELayer:
    return afd.MoELayer(c.H, c.I, c.E, c.k, c.dtype, w, n_shared=c.S, max_tokens=max_tokens,
                        max_sources=max_sources)


def out_to_f64(outs) -> np.ndarray:
    return torch.cat([o.float() for o in outs]).cpu().numpy().astype(np.float64)


def ref_to_f64(c: synth.LayerConfig, ref_out: np.ndarray) -> np.ndarray:
    if c.dtype == "fp32":
        return ref_out.astype(np.float64)
    return oracle.bf16_to_f32(ref_out).astype(np.float64)


def assert_close(c: synth.LayerConfig, got: np.ndarray, exp: np.ndarray):
    tol = TOL[c.dtype]
    den = np.linalg.norm(exp)
    rel = np.linalg.norm(got - exp) / (den if den > 0 else 1.0)
    assert rel <= tol["rel"], f"relative Frobenius error {rel:.3e} > {tol['rel']}"
    if tol["abs"] is not None:
        mx = float(np.abs(got - exp).max()) if got.size else 0.0
        assert mx <= tol["abs"], f"max-abs error {mx:.3e} > {tol['abs']}"
    return rel


def assert_routing_exact(c: synth.LayerConfig, r: dict, ref: dict, T: int):
    """Top-k indices, logits, counts, offsets, permutation and positions bit
    for bit; routing weights within W_ATOL."""
    k, E = c.k, c.E
    idx = r["idx"].cpu().numpy().reshape(T, k)
    assert np.array_equal(idx, ref["idx"]), "top-k indices differ"
    got = r["logits"].cpu().numpy().reshape(T, E)
    if c.dtype == "fp32":  # every logit in the canonical order
        assert np.array_equal(got.view(np.uint32), ref["logits"].view(np.uint32)), "router logits differ"
    else:  # canonical values for every selected expert (others are tensor-core estimates)
        rows = np.arange(T)[:, None]
        assert np.array_equal(got[rows, idx].view(np.uint32), ref["logits"][rows, idx].view(np.uint32)), \
            "selected router logits differ"
    w = r["w"].cpu().numpy().reshape(T, k)
    assert np.abs(w - ref["w"]).max() <= W_ATOL
    counts, offsets, perm, pos = oracle.routing_tables(ref["idx"], E)
    assert np.array_equal(r["counts"].cpu().numpy(), counts)
    assert int(counts.sum()) == T * k
    assert np.array_equal(r["offsets"].cpu().numpy(), offsets)
    assert np.array_equal(r["perm"].cpu().numpy(), perm)
    assert np.array_equal(r["pos"].cpu().numpy(), pos)


def run_case(c: synth.LayerConfig, counts, seed=0, tokens=None, n_micro=1, weights=None, max_tokens=None,
             max_sources=None):
    """Run the CUDA layer and the oracle; returns (layer, srcs, outs, routing, ref)."""
    T = sum(counts)
    srcs = synth.make_sources(c, "cuda", seed=seed, counts=counts)
    w = weights if weights is not None else synth.make_weights(c, "cuda", seed=seed)
    layer = make_layer(c, w, max_tokens=max_tokens or max(T, 1),
                       max_sources=max_sources or max(len(counts), 1))
    outs = layer.forward(srcs, n_micro=n_micro)
    torch.cuda.synchronize()
    layer.check()
    r = layer.routing(T)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(cfg_dict(c), [synth.to_numpy_bits(s) for s in srcs], synth.weights_numpy(w),
                             tokens=tokens)
    return layer, srcs, outs, r, ref
