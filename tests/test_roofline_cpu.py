"""The roofline accounting bench.py reports, pinned to hand-computed values for
the layer's workloads (FLOPs of "MoE系统与AFD架构概述" section 2.1: 6*B*H*I per
expert pass; algorithmic bytes = touched weights once + the layer's own input and
output, staging buffers excluded)."""
from ffn_side_attention_gb300 import roofline, synth


def test_flops_are_six_t_k_h_i():
    c = synth.CONFIGS["qwen3_bf16"]
    assert roofline.layer_flops(c, 3160) == 6 * 3160 * 8 * 4096 * 1536
    assert roofline.gateup_flops(c, 3160) * 3 == roofline.layer_flops(c, 3160) * 2
    d = synth.CONFIGS["dsv3_fp8"]  # one shared expert: k + 1 expert passes per token
    assert roofline.layer_flops(d, 4096) == 6 * 4096 * 9 * 7168 * 2048
    assert roofline.router_flops(d, 4096) == 2 * 4096 * 7168 * 256


def test_bf16_layer_bytes_by_hand():
    c = synth.CONFIGS["qwen3_bf16"]
    w = 3 * 4096 * 1536 * 2            # one expert's three bf16 matrices
    router = 4096 * 128 * 2
    io = 3160 * 4096 * 2 * 2           # x read once, out written once
    assert roofline.layer_bytes(c, 3160, 128) == 128 * w + router + io
    assert roofline.layer_bytes(c, 6, 40) == 40 * w + router + 6 * 4096 * 2 * 2
    rows = 3160 * 8
    assert roofline.gateup_bytes(c, 3160, 128) == 128 * 2 * 4096 * 1536 * 2 + rows * (4096 * 2 + 1536 * 2)
    assert roofline.down_bytes(c, 3160, 128) == 128 * 4096 * 1536 * 2 + rows * (1536 * 2 + 4096 * 2)


def test_fp8_bytes_count_block_scales():
    c = synth.CONFIGS["qwen3_fp8"]
    blocks = (4096 // 128) * (1536 // 128)
    w = 3 * 4096 * 1536 + 3 * blocks * 4          # e4m3 codes + one fp32 scale per 128x128 block
    router = 4096 * 128 * 2                         # the router stays bf16
    io = 1580 * 4096 * 2 * 2                        # bf16 in and out
    assert roofline.layer_bytes(c, 1580, 128) == 128 * w + router + io
    rows = 1580 * 8
    gu = 128 * (2 * 4096 * 1536 + 2 * blocks * 4) + rows * (4096 + 1536) + rows * (4096 // 128 + 1536 // 128) * 4
    assert roofline.gateup_bytes(c, 1580, 128) == gu


def test_t_roof_takes_the_slower_bound():
    t, b = roofline.t_roof(2e12, 1e9, 1000.0, 1000.0)   # 2 ms of compute vs 1 ms of memory
    assert b == "tensor" and abs(t - 2e-3) < 1e-12
    t, b = roofline.t_roof(1e12, 4e9, 1000.0, 1000.0)   # 1 ms vs 4 ms
    assert b == "hbm" and abs(t - 4e-3) < 1e-12
