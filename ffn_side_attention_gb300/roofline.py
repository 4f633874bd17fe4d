"""FLOP and byte accounting of the layer, for the roofline.

FLOPs ("MoE系统与AFD架构概述", section 2.1): a SwiGLU expert pass over B
tokens costs 6*B*H*I FLOPs (three H x I matrices, 2 FLOPs per multiply-add);
with k routed experts and S shared ones per token the layer costs
6*T*(k+S)*H*I.  The router's 2*T*H*E is counted separately.

Bytes are ALGORITHMIC (what a perfect implementation must move through HBM):
the weights of every expert the batch touches, read once (plus FP8 block
scales), and each kernel's own activation inputs/outputs once.  Per unit:
  * touched expert  : gate+up 2*H*I*b_w, down H*I*b_w (+ 4 bytes per
                      128x128 block for fp8)
  * packed row (a routed copy of a token, or a shared-expert row):
      gate/up kernel  : reads H*b_a (+ H/128 scales) and writes I*b_h (+ I/128)
      down kernel     : reads I*b_h (+ I/128) and writes H*2 (bf16 Y)
  * whole layer     : touched experts' weights + shared expert + router
                      weights + T*H*b_in read + T*H*b_out written (the
                      staging buffers P, h, Y are not algorithmic).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Sizes:
    b_w: float    # weight element bytes
    b_a: float    # packed activation element bytes (GEMM B operand of gate/up)
    b_h: float    # SwiGLU output element bytes
    b_y: float    # expert output (Y) element bytes
    b_io: float   # layer input/output element bytes
    scale_blk: bool  # fp8: 4-byte scale per 128 (activations) / 128x128 (weights)


def sizes(dtype: str) -> Sizes:
    if dtype == "fp32":
        return Sizes(4, 4, 4, 4, 4, False)
    if dtype == "bf16":
        return Sizes(2, 2, 2, 2, 2, False)
    return Sizes(1, 1, 1, 2, 2, True)


def layer_flops(cfg, T: int) -> int:
    return 6 * T * (cfg.k + cfg.S) * cfg.H * cfg.I


def router_flops(cfg, T: int) -> int:
    return 2 * T * cfg.H * cfg.E


def _wbytes(cfg, nmats: int) -> float:
    z = sizes(cfg.dtype)
    b = nmats * cfg.H * cfg.I * z.b_w
    if z.scale_blk:
        b += nmats * (cfg.H // 128) * (cfg.I // 128) * 4
    return b


def gateup_bytes(cfg, T: int, touched: int) -> float:
    """Algorithmic bytes of one gate/up + SwiGLU launch."""
    z = sizes(cfg.dtype)
    rows = T * (cfg.k + cfg.S)
    groups = touched + cfg.S
    b = groups * _wbytes(cfg, 2) + rows * (cfg.H * z.b_a + cfg.I * z.b_h)
    if z.scale_blk:
        b += rows * (cfg.H // 128 + cfg.I // 128) * 4
    return b


def gateup_flops(cfg, T: int) -> int:
    """FLOPs of one gate/up launch: two H x I products per packed row."""
    return 4 * T * (cfg.k + cfg.S) * cfg.H * cfg.I


def down_bytes(cfg, T: int, touched: int) -> float:
    z = sizes(cfg.dtype)
    rows = T * (cfg.k + cfg.S)
    groups = touched + cfg.S
    b = groups * _wbytes(cfg, 1) + rows * (cfg.I * z.b_h + cfg.H * z.b_y)
    if z.scale_blk:
        b += rows * (cfg.I // 128) * 4
    return b


def layer_bytes(cfg, T: int, touched: int) -> float:
    z = sizes(cfg.dtype)
    act = 4 if cfg.dtype == "fp32" else 2
    return ((touched + cfg.S) * _wbytes(cfg, 3) + cfg.H * cfg.E * act + T * cfg.H * z.b_io * 2)


def t_roof(flops: float, nbytes: float, peak_tflops: float, peak_gbs: float) -> tuple:
    """(seconds, bound) of the slower of compute and memory."""
    tc = flops / (peak_tflops * 1e12)
    tm = nbytes / (peak_gbs * 1e9)
    return (tm, "hbm") if tm >= tc else (tc, "tensor")
