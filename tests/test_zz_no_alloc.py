"""The allocation-free router entry point (afd_ffn_router_noalloc) against the
full layer's routing and against the CPU oracle.  It exists for callers that
cannot allocate device memory (their pool owns all of HBM, or they sit in a
decode loop where an allocation call may block); they must still get the
layer's exact routing.  Its scratch is one fixed device array sized for
T <= 4096, E <= 256, k <= 16; the cases below reach those limits, take the
fp8 layer's dtype, and call it twice in a row (the array keeps the previous
call's contents).  This file is collected last so a failure here stops a -x
run only after every other test has run."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from ffn_side_attention_gb300 import afd, synth

pytestmark = pytest.mark.gpu

W_ATOL = 2e-6  # routing weights vs the oracle's float64 softmax (the parity tests' tolerance)


def _noalloc(c, srcs, w, T):
    """Two calls in a row through the C ABI; returns both (idx, w) results."""
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    bias_ptr = w["router_bias"].data_ptr() if "router_bias" in w else None
    counts = [int(s.shape[0]) for s in srcs]
    res = []
    for call in range(2):
        idx = torch.full((T * c.k,), -1, dtype=torch.int32, device="cuda")
        wt = torch.full((T * c.k,), float("nan"), dtype=torch.float32, device="cuda")
        rc = afd.afd_ffn_router_noalloc(stream, [s.data_ptr() if s.shape[0] else 0 for s in srcs], counts, c.H,
                                        c.E, c.k, c.dtype, w["w_router"].data_ptr(), bias_ptr, idx.data_ptr(),
                                        wt.data_ptr())
        torch.cuda.synchronize()
        assert rc == 0, f"call {call}: status {rc}"
        res.append((idx, wt))
    return res


def _against_oracle(c, srcs, w, res, T):
    x = torch.cat(srcs)
    xb = synth.to_numpy_bits(x)
    wr = synth.to_numpy_bits(w["w_router"])
    bias = w["router_bias"].cpu().numpy() if "router_bias" in w else None
    logits = oracle.router_logits(xb, wr, "fp32" if c.dtype == "fp32" else "bf16", bias)
    idx_ref, w_ref = oracle.topk(logits, c.k)
    for call, (idx, wt) in enumerate(res):
        assert np.array_equal(idx.cpu().numpy().reshape(T, c.k), idx_ref), f"call {call}: indices differ from the oracle"
        assert np.abs(wt.cpu().numpy().reshape(T, c.k) - w_ref).max() <= W_ATOL, f"call {call}: weights differ"


def _case(c, counts, bias, with_layer=True):
    T = sum(counts)
    srcs = synth.make_sources(c, "cuda", counts=counts)
    w = synth.make_weights(c, "cuda")
    if bias and "router_bias" not in w:
        w["router_bias"] = synth.zipf_bias(c.E, 1.2, "cuda")
    res = _noalloc(c, srcs, w, T)
    _against_oracle(c, srcs, w, res, T)
    if with_layer:
        layer = afd.MoELayer(c.H, c.I, c.E, c.k, c.dtype, w, n_shared=c.S, max_tokens=T, max_sources=len(counts))
        layer.forward(srcs)
        ref = layer.routing(T)
        torch.cuda.synchronize()
        for call, (idx, wt) in enumerate(res):
            assert torch.equal(idx, ref["idx"]), f"call {call}: top-k indices differ from afd_ffn_forward's"
            assert torch.equal(wt, ref["w"]), f"call {call}: weights differ from afd_ffn_forward's"
        layer.close()


@pytest.mark.parametrize("name,counts,bias", [
    ("tiny_fp32", [32, 32], False),
    ("small_bf16", [100, 0, 200], True),
    ("qwen3_bf16", [395] * 4, False),
    ("small_fp8", [150, 0, 7, 300], True),
])
def test_noalloc_router_matches_layer_and_oracle(name, counts, bias):
    if name == "small_bf16":
        c = synth.LayerConfig("small_bf16", H=512, I=256, E=64, k=8, S=0, dtype="bf16", B=0, M=0)
    elif name == "small_fp8":
        c = synth.LayerConfig("small_fp8", H=512, I=128, E=64, k=8, S=1, dtype="fp8", B=0, M=0)
    else:
        c = synth.CONFIGS[name]
    _case(c, counts, bias)


def test_noalloc_router_at_its_limits():
    """T = 4096 tokens, E = 256 experts, k = 16 slots: the scratch array is full (4 MiB
    of logits, 256 tile tickets); Zipf-biased routing so a few experts take most tokens."""
    c = synth.LayerConfig("limits_bf16", H=512, I=128, E=256, k=16, S=0, dtype="bf16", B=0, M=0)
    _case(c, [512] * 8, bias=True)


def test_noalloc_router_dsv3_fp8_full_batch():
    """DeepSeek-V3 fp8 shapes (H = 7168, E = 256, k = 8, Zipf bias) at T = 8 x 512: the
    fp8 layer's dtype (bf16 activations and router weights) at the token limit."""
    c = synth.CONFIGS["dsv3_fp8"]
    _case(c, [c.B] * c.M, bias=True)


def test_noalloc_router_rejects_oversize():
    x = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    out_i = torch.zeros(8, dtype=torch.int32, device="cuda")
    out_w = torch.zeros(8, dtype=torch.float32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (w.data_ptr(), None, out_i.data_ptr(), out_w.data_ptr())
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [4097], 256, 64, 1, "bf16", *args) == afd.AFD_ECAPACITY
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [8], 256, 264, 1, "bf16", *args) == afd.AFD_ECAPACITY
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [8], 256, 64, 17, "bf16", *args) == afd.AFD_ECAPACITY
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [8], 256, 60, 1, "bf16", *args) == afd.AFD_EINVAL
