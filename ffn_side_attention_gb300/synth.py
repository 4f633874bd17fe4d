"""Seeded synthetic inputs for the FFN-server MoE layer.

This module only draws numbers and lays them out in the formats the layer
takes.  It holds none of the layer's arithmetic (no routing, no GEMM, no
activation quantisation) and it serves both the CUDA path and the CPU oracle.

Workloads (shapes after the decode batches the AFD pages discuss):

* ``tiny_fp32``   T=64 in 2 buffers of 32, H=128, I=256, E=8, top-2, fp32.
* ``qwen3_bf16``  Qwen3-235B-A22B-shaped layer: H=4096, I=1536, E=128, top-8,
  bf16; per-instance decode batch B in {6, 48, 197, 395} from M in {1, 4, 8}
  buffers (T = B*M).  B=395 / 197 / 6 are the decode batches at 2K / 4K / 128K
  context in the FastAFD blog's colocated MFU measurement (section 1).
* ``qwen3_fp8``   the same shapes with e4m3 weights (FP32 scale per 128x128
  block) and e4m3 activations (per token, per 128 channels), T = 4*395.
* ``dsv3_fp8``    DeepSeek-V3-shaped: H=7168, I=2048, E=256, top-8 plus one
  shared expert, fp8; T in {512, 2048, 4096} from 8 buffers; router logits
  carry a Zipf(s=1.2) log-bias over a seeded permutation of the experts.
* ``step3_bf16``  Step3-shaped: H=7168, I=5120, E=48, top-3 plus one shared
  expert, bf16; T = 2048 from 8 buffers of 256, run as 3 micro-batches.

Distributions: x ~ N(0,1) and weights ~ N(0, 1/fan_in) (fan_in = H for the
router, gate and up, I for down), rounded to the layer dtype by torch's own
casts.  FP8 weights are stored as e4m3 codes plus one FP32 scale per 128x128
block (scale = block amax / 448, codes = torch's e4m3 cast of w/scale); that
is the weight format the layer is given, not a step of the layer.

Seeds: base seed 0 with sub-seeds x=0, router=1, shared expert=999, expert
e = 1000+e, Zipf permutation=7.  Each expert has its own generator so a single
expert's weights can be re-drawn on any device.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace

import torch


@dataclass(frozen=True)
class LayerConfig:
    name: str
    H: int
    I: int
    E: int
    k: int
    S: int  # shared experts (0 or 1)
    dtype: str  # 'fp32' | 'bf16' | 'fp8'
    B: int  # rows per source buffer
    M: int  # number of source buffers
    zipf_s: float = 0.0
    n_micro: int = 1
    batches: tuple = field(default_factory=tuple)  # other (B, M) cases for tests

    @property
    def T(self) -> int:
        return self.B * self.M

    def with_batch(self, B: int, M: int) -> "LayerConfig":
        return replace(self, B=B, M=M)


CONFIGS = {
    "tiny_fp32": LayerConfig("tiny_fp32", H=128, I=256, E=8, k=2, S=0, dtype="fp32", B=32, M=2),
    "qwen3_bf16": LayerConfig("qwen3_bf16", H=4096, I=1536, E=128, k=8, S=0, dtype="bf16", B=395, M=8,
                              batches=tuple((b, m) for b in (6, 48, 197, 395) for m in (1, 4, 8))),
    "qwen3_fp8": LayerConfig("qwen3_fp8", H=4096, I=1536, E=128, k=8, S=0, dtype="fp8", B=395, M=4),
    "dsv3_fp8": LayerConfig("dsv3_fp8", H=7168, I=2048, E=256, k=8, S=1, dtype="fp8", B=512, M=8,
                            zipf_s=1.2, batches=((64, 8), (256, 8), (512, 8))),
    "step3_bf16": LayerConfig("step3_bf16", H=7168, I=5120, E=48, k=3, S=1, dtype="bf16", B=256, M=8,
                              n_micro=3),
}

SUB_X, SUB_ROUTER, SUB_SHARED, SUB_EXPERT0, SUB_ZIPF = 0, 1, 999, 1000, 7


def _gen(device, seed: int, sub: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + sub)
    return g


def act_torch_dtype(cfg: LayerConfig) -> torch.dtype:
    """Dtype of the source / output buffers (fp8 layers take bf16 activations)."""
    return torch.float32 if cfg.dtype == "fp32" else torch.bfloat16


def make_sources(cfg: LayerConfig, device="cpu", seed: int = 0, counts=None, sub: int = SUB_X):
    """M source buffers of x ~ N(0,1); ``counts`` overrides the per-buffer rows."""
    counts = list(counts) if counts is not None else [cfg.B] * cfg.M
    T = sum(counts)
    g = _gen(device, seed, sub)
    x = torch.randn(max(T, 1), cfg.H, generator=g, device=device, dtype=torch.float32)[:T]
    x = x.to(act_torch_dtype(cfg))
    out, r = [], 0
    for c in counts:
        out.append(x[r:r + c].contiguous())
        r += c
    return out


def _block_fp8(w: torch.Tensor):
    """fp32 [R, C] (R, C multiples of 128) -> (e4m3 codes as uint8 [R, C], scales fp32 [R/128, C/128])."""
    R, Cn = w.shape
    blk = w.reshape(R // 128, 128, Cn // 128, 128)
    amax = blk.abs().amax(dim=(1, 3))
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blk / scale[:, None, :, None]).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return q.reshape(R, Cn).view(torch.uint8), scale.contiguous()


def _one_expert(cfg: LayerConfig, device, seed: int, sub: int):
    g = _gen(device, seed, sub)
    H, I = cfg.H, cfg.I
    wg = torch.randn(H, I, generator=g, device=device) / math.sqrt(H)
    wu = torch.randn(H, I, generator=g, device=device) / math.sqrt(H)
    wd = torch.randn(I, H, generator=g, device=device) / math.sqrt(I)
    if cfg.dtype == "fp32":
        return wg, wu, wd, None, None, None
    if cfg.dtype == "bf16":
        return wg.bfloat16(), wu.bfloat16(), wd.bfloat16(), None, None, None
    (qg, sg), (qu, su), (qd, sd) = _block_fp8(wg), _block_fp8(wu), _block_fp8(wd)
    return qg, qu, qd, sg, su, sd


def make_weights(cfg: LayerConfig, device="cpu", seed: int = 0, experts=None):
    """Weights in the layer's input format.

    Keys: w_router [H,E]; w_gate, w_up [E,H,I]; w_down [E,I,H]; for fp8 also
    s_gate, s_up [E,H/128,I/128], s_down [E,I/128,H/128]; with a shared
    expert sh_gate, sh_up [H,I], sh_down [I,H] (+ sh_s_*); router_bias [E] for
    Zipf-biased layers.  ``experts`` (optional) draws only that subset of the
    routed experts and leaves the others zero (for CPU-side sampling)."""
    H, E = cfg.H, cfg.E
    g = _gen(device, seed, SUB_ROUTER)
    wr = torch.randn(H, E, generator=g, device=device) / math.sqrt(H)
    w = {"w_router": wr.to(act_torch_dtype(cfg))}
    store = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[cfg.dtype]
    w["w_gate"] = torch.zeros(E, H, cfg.I, dtype=store, device=device)
    w["w_up"] = torch.zeros(E, H, cfg.I, dtype=store, device=device)
    w["w_down"] = torch.zeros(E, cfg.I, H, dtype=store, device=device)
    if cfg.dtype == "fp8":
        w["s_gate"] = torch.ones(E, H // 128, cfg.I // 128, device=device)
        w["s_up"] = torch.ones(E, H // 128, cfg.I // 128, device=device)
        w["s_down"] = torch.ones(E, cfg.I // 128, H // 128, device=device)
    for e in (range(E) if experts is None else experts):
        qg, qu, qd, sg, su, sd = _one_expert(cfg, device, seed, SUB_EXPERT0 + e)
        w["w_gate"][e], w["w_up"][e], w["w_down"][e] = qg, qu, qd
        if cfg.dtype == "fp8":
            w["s_gate"][e], w["s_up"][e], w["s_down"][e] = sg, su, sd
    if cfg.S:
        qg, qu, qd, sg, su, sd = _one_expert(cfg, device, seed, SUB_SHARED)
        w["sh_gate"], w["sh_up"], w["sh_down"] = qg, qu, qd
        if cfg.dtype == "fp8":
            w["sh_s_gate"], w["sh_s_up"], w["sh_s_down"] = sg, su, sd
    if cfg.zipf_s:
        w["router_bias"] = zipf_bias(E, cfg.zipf_s, device, seed)
    return w


def zipf_bias(E: int, s: float, device="cpu", seed: int = 0) -> torch.Tensor:
    """bias[e] = -s * ln(pi(e) + 1) for a seeded permutation pi of the experts:
    adding it to the logits multiplies each expert's softmax weight by a
    Zipf(s) pmf over the permuted expert ranks."""
    g = _gen("cpu", seed, SUB_ZIPF)
    perm = torch.randperm(E, generator=g)
    return (-s * torch.log(perm.double() + 1.0)).float().to(device)


def to_numpy_bits(t: torch.Tensor):
    """Tensor -> numpy in the oracle's convention (bf16 as uint16 bits, fp8 as uint8 codes)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view("uint16")
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.numpy()


def weights_numpy(w: dict) -> dict:
    return {k: to_numpy_bits(v) for k, v in w.items()}

