"""The allocation-free router entry point (afd_ffn_router_noalloc) against the
full layer's routing.  It exists for callers that cannot allocate device
memory (their pool owns all of HBM, or they sit in a decode loop where an
allocation call may block); they must still get the layer's exact routing.
This file is collected last so a failure here stops a -x run only after every
other test has run."""
import ctypes as C

import pytest
import torch

from ffn_side_attention_gb300 import afd, synth

pytestmark = pytest.mark.gpu

W_ATOL = 2e-6  # the routing-weight tolerance of the parity tests


def _case(c, counts, bias):
    T = sum(counts)
    srcs = synth.make_sources(c, "cuda", counts=counts)
    w = synth.make_weights(c, "cuda")
    if bias and "router_bias" not in w:
        w["router_bias"] = synth.zipf_bias(c.E, 1.2, "cuda")
    layer = afd.MoELayer(c.H, c.I, c.E, c.k, c.dtype, w, n_shared=c.S, max_tokens=T, max_sources=len(counts))
    layer.forward(srcs)
    ref = layer.routing(T)
    torch.cuda.synchronize()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    bias_ptr = w["router_bias"].data_ptr() if "router_bias" in w else None
    for call in range(2):  # two calls in a row share the scratch array
        idx = torch.full((T * c.k,), -1, dtype=torch.int32, device="cuda")
        wt = torch.full((T * c.k,), float("nan"), dtype=torch.float32, device="cuda")
        rc = afd.afd_ffn_router_noalloc(stream, [s.data_ptr() if s.shape[0] else 0 for s in srcs], counts, c.H, c.E,
                                        c.k, c.dtype, w["w_router"].data_ptr(), bias_ptr, idx.data_ptr(),
                                        wt.data_ptr())
        torch.cuda.synchronize()
        assert rc == 0, f"call {call}: status {rc}"
        assert torch.equal(idx, ref["idx"]), f"call {call}: top-k indices differ from afd_ffn_forward's"
        assert (wt - ref["w"]).abs().max().item() <= W_ATOL, f"call {call}: weights differ"
    layer.close()


@pytest.mark.parametrize("name,counts,bias", [
    ("tiny_fp32", [32, 32], False),
    ("small_bf16", [100, 0, 200], True),
    ("qwen3_bf16", [395] * 4, False),
])
def test_noalloc_router_matches_layer_routing(name, counts, bias):
    if name == "small_bf16":
        c = synth.LayerConfig("small_bf16", H=512, I=256, E=64, k=8, S=0, dtype="bf16", B=0, M=0)
    else:
        c = synth.CONFIGS[name]
    _case(c, counts, bias)


def test_noalloc_router_rejects_oversize():
    x = torch.zeros(8, 256, dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(256, 64, dtype=torch.bfloat16, device="cuda")
    out_i = torch.zeros(8, dtype=torch.int32, device="cuda")
    out_w = torch.zeros(8, dtype=torch.float32, device="cuda")
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = (w.data_ptr(), None, out_i.data_ptr(), out_w.data_ptr())
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [4097], 256, 64, 1, "bf16", *args) == afd.AFD_ECAPACITY
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [8], 256, 264, 1, "bf16", *args) == afd.AFD_ECAPACITY
    assert afd.afd_ffn_router_noalloc(stream, [x.data_ptr()], [8], 256, 60, 1, "bf16", *args) == afd.AFD_EINVAL
