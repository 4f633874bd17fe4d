"""GPU parity: the CUDA layer (through the C ABI) against the CPU oracle on
the same seeded inputs.  Routing is compared bit for bit; outputs within the
dtype's tolerance (tests/gpu_helpers.py)."""
import numpy as np
import pytest
import torch

from ffn_side_attention_gb300 import afd, synth

import oracle
from gpu_helpers import (assert_close, assert_routing_exact, cfg_dict, make_layer, out_to_f64, ref_to_f64, run_case)

pytestmark = pytest.mark.gpu


def _small(dtype="bf16", H=256, I=256, E=16, k=4, S=0, zipf=0.0):
    return synth.LayerConfig("small", H=H, I=I, E=E, k=k, S=S, dtype=dtype, B=0, M=0, zipf_s=zipf)


def test_tiny_fp32_layer():
    c = synth.CONFIGS["tiny_fp32"]
    layer, srcs, outs, r, ref = run_case(c, [c.B] * c.M)
    assert_routing_exact(c, r, ref, c.T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


@pytest.mark.parametrize("shape,counts", [
    (dict(), [17, 0, 40]),                                   # ragged, an empty buffer
    (dict(S=1), [1]),                                        # single token + shared expert
    (dict(E=4, k=2, H=512, I=384), [300, 301]),              # experts with > 256 rows: several N tiles
    (dict(E=64, k=8, H=768, I=640, S=1), [5, 3, 0, 9]),      # many experts, few tokens
    (dict(E=8, k=8, H=256, I=128), [33]),                    # k = E: every expert on every token
    (dict(E=8, k=1), [40, 3]),                               # k = 1: one slot, weight 1
    (dict(E=1, k=1, S=1), [20]),                             # one routed expert (and the shared one)
])
def test_bf16_shapes(shape, counts):
    c = _small(**shape)
    T = sum(counts)
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert_routing_exact(c, r, ref, T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_largest_router_and_source_table(dtype):
    """The configuration limits at once: E = 256 experts plus a shared one (257 groups),
    k = 16 slots, and M = 64 source buffers with empty ones among them; batches on both
    router paths (small-batch kernel, and the tensor-core estimate with exact candidates)."""
    c = _small(dtype=dtype, E=256, k=16, H=256, I=128, S=1)
    rng = np.random.default_rng(3)
    for counts in ([int(v) for v in rng.integers(0, 3, 64)], [int(v) for v in rng.integers(0, 40, 64)]):
        layer, srcs, outs, r, ref = run_case(c, counts, max_sources=64)
        assert_routing_exact(c, r, ref, sum(counts))
        assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))
        layer.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_tensor_core_router_tiles_per_source(dtype):
    """The tensor-core router reads its 128-token tiles from each source buffer in place:
    sources of 300, 0, 129, 1 and 77 rows give tiles that end mid-source, a source of one
    row, and an empty source between two others (507 tokens, 128 experts: the estimate
    path)."""
    c = _small(dtype=dtype, E=128, k=8, H=256, I=128)
    counts = [300, 0, 129, 1, 77]
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert layer.launches_per_forward(sum(counts)) == 7  # two router launches: not the small path
    assert_routing_exact(c, r, ref, sum(counts))
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


def test_bf16_zipf_bias_imbalance():
    """Zipf(1.2) log-bias on the logits: a few experts take most tokens."""
    c = _small(E=64, k=8, H=512, I=256, zipf=1.2)
    counts = [100, 100, 100]
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert_routing_exact(c, r, ref, 300)
    assert r["counts"].max().item() > 256  # the hot expert spans two token tiles
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


@pytest.fixture(scope="module")
def qwen3_bf16_layer():
    """One qwen3_bf16 layer (H=4096, I=1536, E=128, k=8) sized for the largest aggregated
    batch (8 x 395 tokens), shared by the twelve (B, M) decode-batch cases."""
    c = synth.CONFIGS["qwen3_bf16"]
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=c.T, max_sources=c.M)
    yield c, layer, synth.weights_numpy(w)
    layer.close()


@pytest.mark.parametrize("B,M", list(synth.CONFIGS["qwen3_bf16"].batches))
def test_qwen3_bf16_every_decode_batch_full_output(qwen3_bf16_layer, B, M):
    """Every (B, M) point of the Qwen3 bf16 workload: per-instance decode batches
    B in {6, 48, 197, 395} (FastAFD blog section 1) aggregated from M in {1, 4, 8}
    attention instances (section 2).  Routing bit-exact and the WHOLE output within the
    bf16 tolerance of the oracle, up to T = 3160."""
    base, layer, wn = qwen3_bf16_layer
    c = base.with_batch(B, M)
    srcs = synth.make_sources(c, "cuda", seed=B * 10 + M)
    outs = layer.forward(srcs)
    torch.cuda.synchronize()
    layer.check()
    r = layer.routing(c.T)
    torch.cuda.synchronize()
    ref = oracle.moe_forward(cfg_dict(c), [synth.to_numpy_bits(s) for s in srcs], wn)
    assert_routing_exact(c, r, ref, c.T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


def test_pipelined_equals_single_and_deterministic():
    c = _small(E=16, k=4, S=1, H=512, I=256)
    counts = [50, 0, 77, 12]
    srcs = synth.make_sources(c, "cuda", counts=counts)
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=200, max_sources=8)
    a = [o.clone() for o in layer.forward(srcs)]
    b = [o.clone() for o in layer.forward(srcs)]
    for n in (2, 3, 4):
        p = layer.forward(srcs, n_micro=n)
        torch.cuda.synchronize()
        for x, y in zip(a, p):
            assert torch.equal(x, y), f"pipelined n_micro={n} differs"
    for x, y in zip(a, b):
        assert torch.equal(x, y), "two forwards differ"
    layer.check()


def test_fp8_pipelined_equals_single_pass():
    """The fp8 layer micro-batched in 2, 3 and 4 parts gives the single pass bit for bit:
    activations are quantised per token, every MMA row is one token's, the promotion scale
    and the re-quantisation of h are per token, and the combine sums each token's slots in
    order, so how tokens share tiles changes nothing.  The single pass matches the oracle."""
    c = _small(dtype="fp8", E=16, k=4, S=1, H=512, I=256)
    counts = [50, 0, 77, 12]
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))
    single = [o.clone() for o in outs]
    for n in (2, 3, 4):
        p = layer.forward(srcs, n_micro=n)
        torch.cuda.synchronize()
        for x, y in zip(single, p):
            assert torch.equal(x, y), f"fp8 n_micro={n} differs from the single pass"
    layer.check()
    layer.close()


@pytest.mark.parametrize("counts,n_micro", [([9, 0, 8], 2), ([4, 21], 3), ([33], 4)])
def test_pipelined_mixes_packed_and_direct_micro_batches(counts, n_micro):
    """Micro-batches on both sides of the pack-free limit (8 bf16 tokens) in one forward:
    17 tokens in 9 + 8, 25 in 9 + 8 + 8, 33 in 9 + 8 + 8 + 8.  The first micro-batch's
    gate/up reads the packed rows, the others' read the sources; the outputs equal the
    single pass bit for bit, and the oracle within the bf16 tolerance."""
    c = _small(E=16, k=4, S=1, H=512, I=256)
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))
    single = [o.clone() for o in outs]
    for _ in range(2):
        p = layer.forward(srcs, n_micro=n_micro)
        torch.cuda.synchronize()
        for x, y in zip(single, p):
            assert torch.equal(x, y), f"n_micro={n_micro} differs from the single pass"
    layer.check()
    layer.close()


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_outputs_follow_their_tokens(dtype):
    """Per-token independence on the GPU: permuting tokens within and across the source
    buffers (and changing how many buffers carry them) permutes the outputs bit for bit."""
    c = _small(dtype=dtype, E=16, k=4, H=256, I=256, S=1)
    counts = [37, 0, 91]
    srcs = synth.make_sources(c, "cuda", seed=5, counts=counts)
    w = synth.make_weights(c, "cuda", seed=5)
    layer = make_layer(c, w, max_tokens=160, max_sources=4)
    x = torch.cat(srcs)
    y = torch.cat(layer.forward(srcs)).clone()
    torch.cuda.synchronize()
    perm = torch.randperm(x.shape[0], generator=torch.Generator().manual_seed(11)).to(x.device)
    xp = x[perm]
    regrouped = [xp[:50].contiguous(), xp[50:51].contiguous(), xp[51:].contiguous()]
    yp = torch.cat(layer.forward(regrouped))
    torch.cuda.synchronize()
    layer.check()
    assert torch.equal(yp, y[perm])


def test_forward_host_equals_device():
    c = _small(E=16, k=4, H=256, I=256)
    counts = [20, 9]
    srcs = synth.make_sources(c, "cuda", counts=counts)
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=64, max_sources=4)
    dev = layer.forward(srcs)
    torch.cuda.synchronize()
    hs = [s.cpu().pin_memory() for s in srcs]
    ho = [torch.empty_like(s).pin_memory() for s in hs]
    layer.forward_host(hs, ho)
    for x, y in zip(dev, ho):
        assert torch.equal(x.cpu(), y)
    # the pipelined path through host buffers equals the single pass bit for bit
    ho3 = [torch.empty_like(s).pin_memory() for s in hs]
    layer.forward_host(hs, ho3, n_micro=3)
    for x, y in zip(dev, ho3):
        assert torch.equal(x.cpu(), y)
    with pytest.raises(afd.AfdError):
        layer.forward_host(hs, ho3, n_micro=0)


@pytest.mark.parametrize("n_micro,E,dtype", [([1] * 5, 16, "bf16"), ([3] * 5, 16, "bf16"),
                                             ([1, 3, 1, 1, 2], 16, "bf16"), ([1] * 5, 128, "bf16"),
                                             ([1, 2, 1, 1, 3], 128, "bf16"), ([1, 3, 1, 1, 2], 16, "fp8")])
def test_forward_host_async_stream_of_batches(n_micro, E, dtype):
    """Consecutive asynchronous host-buffer calls (staging slots reused every other
    call, single-pass calls alternating compute streams and workspaces, batch sizes
    and micro-batch counts changing) give, call by call, the device forward's outputs;
    afterwards the routing read-out is the last call's.  With 128 experts the larger
    batches take the tensor-core router, whose source tensor maps then follow the
    staging slots from call to call.  One case runs the fp8 layer (quantising pack)."""
    c = _small(dtype=dtype, E=E, k=4, H=256, I=256, S=1)
    w = synth.make_weights(c, "cuda")
    big = E == 128
    layer = make_layer(c, w, max_tokens=320 if big else 96, max_sources=4)
    batches = ([[300, 9], [33, 200, 40], [5], [160, 160], [1, 250, 3]] if big else
               [[20, 9], [33, 0, 40], [5], [48, 48], [1, 2, 3]])
    expect, hin, hout = [], [], []
    for i, counts in enumerate(batches):
        srcs = synth.make_sources(c, "cuda", seed=10 + i, counts=counts)
        expect.append([o.cpu() for o in layer.forward(srcs)])
        torch.cuda.synchronize()
        hin.append([x.cpu().pin_memory() for x in srcs])
        hout.append([torch.full_like(x, float("nan")).pin_memory() for x in hin[-1]])
    T_last = sum(batches[-1])
    r_expect = {k: v.clone() for k, v in layer.routing(T_last).items()}
    torch.cuda.synchronize()  # the library streams do not wait for torch's stream
    for i in range(len(batches)):
        layer.forward_host_async(hin[i], hout[i], n_micro=n_micro[i])
    layer.host_wait()
    for i in range(len(batches)):
        for x, y in zip(expect[i], hout[i]):
            assert torch.equal(x, y), f"call {i}"
    if n_micro[-1] == 1:
        r = layer.routing(T_last)
        for k in ("idx", "w", "counts", "offsets", "perm", "pos"):
            assert torch.equal(r[k], r_expect[k]), k
    with pytest.raises(afd.AfdError):
        layer.forward_host_async(hin[0], hout[0], n_micro=0)
    layer.host_wait()
    layer.check()


@pytest.mark.parametrize("kind,text", [(afd.INJECT_TIMEOUT, r"word 0x1: a bounded wait timed out;$"),
                                       (afd.INJECT_RANGE, r"word 0x2: a routing value was out of range;$")])
def test_device_checks_report_and_the_handle_recovers(kind, text):
    """A bounded wait that runs out (nothing ever arrives; the wait gives up after ~1 ms)
    and an out-of-range expert id in the routing tables each set the device error word,
    afd_ffn_check reports it, and the next forward on the same handle is clean and
    unchanged."""
    c = _small(E=16, k=4, H=256, I=256)
    counts = [20, 9]
    srcs = synth.make_sources(c, "cuda", counts=counts)
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=64, max_sources=4)
    before = torch.cat(layer.forward(srcs)).clone()
    layer.check()
    layer.debug_inject(kind, 2_000_000)
    with pytest.raises(afd.AfdError, match=text):
        layer.check()
    after = torch.cat(layer.forward(srcs))
    layer.check()
    assert torch.equal(before, after)
    with pytest.raises(afd.AfdError):
        layer.debug_inject(7)


def test_launches_per_forward_by_batch():
    """One router launch for small batches (up to 152 tokens with 128 experts), two
    (tensor-core logits, select) for larger ones; routing tables in one launch up to 2048
    tokens (a warp, a block, or blocks that each count the whole batch) and two above;
    then pack (none up to 8 tokens: the gate/up GEMM reads the sources), 2 GEMMs,
    combine."""
    c = synth.CONFIGS["qwen3_bf16"]
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=4096, max_sources=8)
    assert layer.launches_per_forward(6) == 5
    assert layer.launches_per_forward(8) == 5     # last batch without a pack launch
    assert layer.launches_per_forward(9) == 6
    assert layer.launches_per_forward(152) == 6   # last batch of the single-launch router
    assert layer.launches_per_forward(160) == 7   # two router launches, one routing launch
    assert layer.launches_per_forward(2048) == 7
    assert layer.launches_per_forward(2049) == 8  # two routing launches above 2048 tokens
    assert layer.launches_per_forward(3160) == 8
    with pytest.raises(afd.AfdError):
        layer.launches_per_forward(0)


@pytest.mark.parametrize("counts", [[1] * 8, [0, 3, 1, 0, 4], [2] * 4 + [1], [8]])
def test_bf16_gateup_reads_the_sources_up_to_8_tokens(counts):
    """bf16 batches of at most 8 tokens run no pack: the gate/up GEMM's token producer copies
    each packed row from its token's own source buffer (one lane per row, one-row tensor
    maps).  Covered: 8 one-token sources, ragged sources with empty ones, 9 tokens (the
    packed form, just past the limit), and one source whose 8 tokens all reach the shared
    expert and, with 4 experts and k = 4, every routed one (every group at the limit).
    Routing bit-exact and the full output against the oracle."""
    c = _small(E=4 if counts == [8] else 16, k=4, H=512, I=256, S=1)
    T = sum(counts)
    layer, srcs, outs, r, ref = run_case(c, counts, max_sources=64)
    assert layer.launches_per_forward(T) == (5 if T <= 8 else 6)
    assert_routing_exact(c, r, ref, T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))
    layer.close()


@pytest.mark.parametrize("counts", [[1], [31, 1], [32, 1], [255, 1], [256, 1], [1000, 24], [2000, 48],
                                    [2048, 1], [20000, 20001]])
def test_routing_tables_edges(counts):
    """Routing tables at the boundaries of their forms: one warp up to 32 tokens, one block
    up to 256, one launch of blocks that each count the whole batch up to 2048, two
    launches above (32/33, 256/257, 1024, 2048/2049 tokens, and 40001 tokens in 157
    blocks).  Tables bit-exact against the oracle, and identical on several forwards in a
    row."""
    c = _small(E=16, k=4, H=256, I=128, S=1)
    layer, srcs, outs, r, ref = run_case(c, counts)
    T = sum(counts)
    assert_routing_exact(c, r, ref, T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))
    for _ in range(3):
        again = layer.forward(srcs)
        torch.cuda.synchronize()
        layer.check()
        r2 = layer.routing(T)
        for key in ("counts", "offsets", "perm", "pos"):
            assert torch.equal(r2[key], r[key]), key
        for x, y in zip(outs, again):
            assert torch.equal(x, y)


@pytest.mark.parametrize("dtype,n_micro,E,counts", [
    ("bf16", 1, 16, [300, 0, 250]), ("fp8", 1, 16, [300, 0, 250]), ("bf16", 3, 16, [300, 0, 250]),
    ("bf16", 1, 128, [300, 0, 250]), ("fp8", 1, 128, [300, 0, 250]),
    ("bf16", 1, 16, [5, 0, 3]), ("bf16", 3, 128, [5, 0, 3])])  # no pack: the GEMM reads the sources
def test_forward_captured_in_a_cuda_graph_replays_like_eager(dtype, n_micro, E, counts):
    """afd_ffn_forward enqueues no host synchronisation and keeps no per-launch host state
    on the device path, so a serving loop can capture it in a CUDA graph: replaying the
    graph over new contents of the captured source buffers gives, each time, the eager
    forward's outputs bit for bit (550 tokens: the one-launch routing tables for more than
    256 tokens; 8 tokens: no pack).  With micro-batches the capture spans the library's own
    streams, forked from and joined back to the capturing stream with events.  With 128
    experts at 550 tokens the router takes the tensor-core path, and at 8 bf16 tokens the
    gate/up GEMM reads the sources: both through source tensor maps passed as kernel
    parameters.  The eager forwards in between run on other buffers (the library encodes
    their maps), and each replay still reads the captured buffers."""
    c = _small(dtype=dtype, E=E, k=4, H=256, I=256, S=1)
    T = sum(counts)
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=600, max_sources=4)
    router = 2 if E == 128 and T > 152 else 1  # tensor-core logits + select, or the small-batch kernel
    pack = 0 if dtype == "bf16" and T <= 8 else 1
    assert layer.launches_per_forward(T) == router + 1 + pack + 2 + 1  # routing, pack, GEMMs, combine
    static_in = synth.make_sources(c, "cuda", seed=1, counts=counts)
    static_out = [torch.empty_like(x) for x in static_in]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        layer.forward(static_in, static_out, n_micro=n_micro)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer.forward(static_in, static_out, n_micro=n_micro)
    for seed in (2, 3, 4):
        fresh = synth.make_sources(c, "cuda", seed=seed, counts=counts)
        for dst, src in zip(static_in, fresh):
            dst.copy_(src)
        graph.replay()
        torch.cuda.synchronize()
        eager = layer.forward(fresh)
        torch.cuda.synchronize()
        for x, y in zip(static_out, eager):
            assert torch.equal(x, y), f"replay with inputs {seed} differs from the eager forward"
    layer.check()
    layer.close()


def test_empty_batch_is_noop():
    c = _small()
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=8, max_sources=4)
    srcs = [torch.empty(0, c.H, dtype=torch.bfloat16, device="cuda")] * 3
    outs = layer.forward(srcs)
    layer.check()
    assert all(o.shape[0] == 0 for o in outs)


def test_argument_errors():
    c = _small()
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=8, max_sources=2)
    x = synth.make_sources(c, "cuda", counts=[9])
    with pytest.raises(afd.AfdError) as e:
        layer.forward(x)
    assert e.value.code == afd.AFD_ECAPACITY
    x = synth.make_sources(c, "cuda", counts=[1, 1, 1])
    with pytest.raises(afd.AfdError) as e:
        layer.forward(x)
    assert e.value.code == afd.AFD_ECAPACITY
    big = torch.zeros(3 * c.H + 8, dtype=torch.bfloat16, device="cuda")
    mis = big[1:1 + 2 * c.H].view(2, c.H)  # 2-byte offset: not 16-byte aligned
    with pytest.raises(afd.AfdError) as e:
        layer.forward([mis])
    assert e.value.code == afd.AFD_EINVAL
    with pytest.raises(afd.AfdError) as e:
        layer.forward(x[:1], n_micro=9)
    assert e.value.code == afd.AFD_EINVAL
    layer.check()


@pytest.mark.parametrize("shape,counts", [
    (dict(H=264, I=128, E=12, k=3), [7, 30]),     # partial 256-channel slab, partial expert tile
    (dict(H=8, I=16, E=5, k=5), [3]),             # one chunk of channels, k = E
])
def test_fp32_router_edges(shape, counts):
    c = _small(dtype="fp32", **shape)
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert_routing_exact(c, r, ref, sum(counts))
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


@pytest.mark.parametrize("shape,counts", [
    (dict(dtype="fp8", S=1), [17, 0, 40]),
    (dict(dtype="fp8", E=4, k=2, H=512, I=384), [300, 301]),       # > 128 rows per expert: several N tiles
    (dict(dtype="fp8", E=48, k=3, H=768, I=640, S=1), [2, 5]),
    (dict(dtype="fp8", E=8, k=1), [50]),                          # k = 1
    (dict(dtype="fp8", E=4, k=2, H=7424, I=256), [40]),            # 58 K blocks in gate/up
    (dict(dtype="fp8", E=4, k=2, H=256, I=7296, S=1), [40]),       # 57 K blocks in down
])
def test_fp8_shapes(shape, counts):
    c = _small(**shape)
    layer, srcs, outs, r, ref = run_case(c, counts)
    assert_routing_exact(c, r, ref, sum(counts))
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


@pytest.mark.parametrize("T", [1, 32, 33, 64, 65, 127, 160, 193])
def test_fp8_tile_fill_at_the_short_tile_bounds(T):
    """k = E: every expert (and the shared one) gets all T tokens, so the last tile of each
    group holds T mod 128 rows (128 when that is 0): tiles filled to 1, 32, 33, 64, 65 and
    127 rows exercise the TMA boxes of 32 token rows and the epilogue warps whose lanes
    hold no token."""
    c = _small(dtype="fp8", E=8, k=8, H=512, I=256, S=1)
    layer, srcs, outs, r, ref = run_case(c, [T])
    assert_routing_exact(c, r, ref, T)
    assert np.all(r["counts"].cpu().numpy() == T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


def _sampled(c, n_random=12, seed=13):
    T = c.T
    rng = np.random.default_rng(seed)
    edges = {0, T - 1} | {m * c.B for m in range(c.M)} | {m * c.B - 1 for m in range(1, c.M)}
    return sorted(edges | set(rng.choice(T, n_random, replace=False).tolist()))


def test_qwen3_fp8_full_output():
    """qwen3_fp8 at its full size (T = 4 x 395): the whole output against the oracle."""
    c = synth.CONFIGS["qwen3_fp8"]
    layer, srcs, outs, r, ref = run_case(c, [c.B] * c.M)
    assert_routing_exact(c, r, ref, c.T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


@pytest.mark.parametrize("B", [64, 256, 512])
def test_dsv3_fp8_zipf(B):
    """DeepSeek-V3 shapes, Zipf-biased routing, shared expert; T = 8 x B.  T = 512: the
    whole output; T = 2048 and 4096 (oracle minutes per full pass): routing on every
    token, outputs on 64 sampled tokens (buffer edges + random)."""
    c = synth.CONFIGS["dsv3_fp8"].with_batch(B, 8)
    tokens = None if B == 64 else _sampled(c, n_random=48)
    layer, srcs, outs, r, ref = run_case(c, [c.B] * c.M, tokens=tokens)
    assert_routing_exact(c, r, ref, c.T)
    got = out_to_f64(outs) if tokens is None else out_to_f64(outs)[tokens]
    assert_close(c, got, ref_to_f64(c, ref["out"]))


def test_step3_bf16_three_microbatches_sampled():
    """Step3 shapes: T = 8 x 256 as three pipelined micro-batches (683/683/682),
    bitwise equal to one pass, sampled tokens against the oracle."""
    c = synth.CONFIGS["step3_bf16"]
    tokens = _sampled(c, n_random=48)
    layer, srcs, outs, r, ref = run_case(c, [c.B] * c.M, tokens=tokens)
    assert_routing_exact(c, r, ref, c.T)
    assert_close(c, out_to_f64(outs)[tokens], ref_to_f64(c, ref["out"]))
    piped = layer.forward(srcs, n_micro=3)
    torch.cuda.synchronize()
    for x, y in zip(outs, piped):
        assert torch.equal(x, y)


def test_small_batch_router_logits_all_canonical():
    """Small batches (a router grid of at most two waves: up to 152 tokens with 128
    experts) compute every logit in the canonical order with no tensor-core estimate: all
    T*E logits equal the oracle's bit for bit.  T = 152 is the last batch on that path."""
    c = synth.CONFIGS["qwen3_bf16"].with_batch(76, 2)
    layer, srcs, outs, r, ref = run_case(c, [c.B] * c.M)
    got = r["logits"].cpu().numpy().reshape(c.T, c.E)
    assert np.array_equal(got.view(np.uint32), ref["logits"].view(np.uint32))
    assert_routing_exact(c, r, ref, c.T)
    assert_close(c, out_to_f64(outs), ref_to_f64(c, ref["out"]))


def _router_splits(H, E, counts, num_sms):
    """K splits of the tensor-core router logits, as the launcher chooses them: token tiles
    of 128 rows within each source (a tile never spans two sources)."""
    tiles = sum(-(-c // 128) for c in counts) * -(-E // 128)
    num_kb = H // 64
    splits = min(max(1, num_sms // tiles), max(num_kb // 4, 1), 8)
    per = -(-num_kb // splits)
    return -(-num_kb // per)


GUARD_BAND_CASES = [
    ("qwen3_bf16", 395, 2, 1),
    ("qwen3_bf16", 395, 8, 1),
    ("qwen3_fp8", 395, 4, 1),
    ("dsv3_fp8", 64, 8, 1),
    ("dsv3_fp8", 256, 8, 1),
    ("dsv3_fp8", 512, 8, 1),
    ("step3_bf16", 256, 8, 1),
]


@pytest.mark.parametrize("name,B,M,n_micro", GUARD_BAND_CASES)
def test_tensor_core_router_error_within_guard_band(name, B, M, n_micro):
    """The tensor-core logit estimates that are not recomputed exactly must lie within the
    bound the candidate rule assumes, b_e = g * ||x|| * ||w_e|| + 2^-22 (|L~| + |bias|),
    g = (g_canonical + (H/8 + splits + 2) * 2^-21) * 1.0001, with the norms rounded up as the
    kernels round them.  Every shape the layer runs on the estimate path: qwen3 at T = 790
    and 3160, qwen3 fp8, DeepSeek-V3 fp8 with the Zipf bias (H = 7168, E = 256) at its
    three batches, and Step3 (H = 7168, E = 48, k = 3) in one 2048-token pass (its 683-token
    micro-batches take the same estimate path; the read-out covers the first micro-batch).  The
    worst ratio must stay below 1/8 (the 2^-21 per 8 products in g is itself conservative);
    selection and the selected logits are bit-exact against the oracle's canonical ones."""
    c = synth.CONFIGS[name].with_batch(B, M)
    T, E = c.T, c.E
    srcs = synth.make_sources(c, "cuda")
    w = synth.make_weights(c, "cuda")
    layer = make_layer(c, w, max_tokens=T, max_sources=M)
    x = torch.cat(srcs)
    q, rem = divmod(T, n_micro)
    T0 = q + (1 if rem else 0)  # the routing read-out is the first micro-batch's
    layer.forward(srcs, n_micro=n_micro)
    torch.cuda.synchronize()
    layer.check()
    r = layer.routing(T0)
    torch.cuda.synchronize()
    xb = synth.to_numpy_bits(x[:T0])
    wr = synth.to_numpy_bits(w["w_router"])
    bias = w["router_bias"].cpu().numpy() if "router_bias" in w else None
    exact = oracle.router_logits(xb, wr, "bf16", bias)
    idx_ref, w_ref = oracle.topk(exact, c.k)
    idx = r["idx"].cpu().numpy().reshape(T0, c.k)
    assert np.array_equal(idx, idx_ref), "top-k indices differ"
    got32 = r["logits"].cpu().numpy().reshape(T0, E)
    rows = np.arange(T0)[:, None]
    assert np.array_equal(got32[rows, idx].view(np.uint32), exact[rows, idx].view(np.uint32))
    assert np.abs(r["w"].cpu().numpy().reshape(T0, c.k) - w_ref).max() <= 2e-6
    got = got32.astype(np.float64)
    ex = exact.astype(np.float64)
    xf = x[:T0].float().cpu().numpy().astype(np.float64)
    wf = w["w_router"].float().cpu().numpy().astype(np.float64)
    xn = np.linalg.norm(xf, axis=1) * (1 + 1 / 1024)
    wn = np.linalg.norm(wf, axis=0) * (1 + 1 / 1024)
    u = 2.0 ** -24
    n = c.H / 32 + 6
    assert n_micro == 1  # the split count below is for the whole batch's sources
    ns = _router_splits(c.H, E, [c.B] * c.M, torch.cuda.get_device_properties(0).multi_processor_count)
    g = (n * u / (1 - n * u) + (c.H / 8 + ns + 2) * 2.0 ** -21) * 1.0001
    babs = np.abs(bias.astype(np.float64))[None, :] if bias is not None else 0.0
    bound = g * xn[:, None] * wn[None, :] + 2.0 ** -22 * (np.abs(got) + babs)
    est = got32.view(np.uint32) != exact.view(np.uint32)  # entries holding the tensor-core estimate
    assert est.sum() > T0 * E // 2  # most entries are estimates
    ratio = np.abs(got - ex)[est] / bound[est]
    # the candidate rule, replayed: experts whose upper end reaches the k-th largest lower end
    lo = np.sort(got - bound, axis=1)[:, -c.k]
    ncand = (got + bound >= lo[:, None]).sum(axis=1)
    print(f"guard band {name} T={T} n_micro={n_micro}: worst ratio {ratio.max():.3e}, "
          f"candidates per token {ncand.mean():.2f} (max {ncand.max()})")
    assert ratio.max() < 1 / 8, f"tensor-core error reached {ratio.max():.3f} of the guard band"
    layer.close()
