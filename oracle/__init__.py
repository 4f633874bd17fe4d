"""CPU oracle for the AFD FFN-server MoE layer (test infrastructure only).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product library never loads it and
shares no code with it.  The arithmetic lives in ``afd_oracle.c`` (plain C,
OpenMP over tokens, fp64 accumulation); this module only marshals numpy
arrays into it.

bf16 tensors cross this boundary as ``np.uint16`` bit patterns, e4m3 as
``np.uint8`` codes.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "afd_oracle.c")
_SO = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

FP32, BF16, FP8 = 0, 1, 2
DTYPES = {"fp32": FP32, "bf16": BF16, "fp8": FP8}


def build(force: bool = False) -> str:
    """Compile afd_oracle.c into liboracle.so with gcc (no -ffast-math, no FMA
    contraction: the oracle's rounding must be exactly what the C says)."""
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(_SRC):
        tmp = _SO + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.check_call(cmd)
        os.replace(tmp, _SO)
    return _SO


class _Cfg(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int),
                ("n_shared", C.c_int), ("dtype", C.c_int)]


class _Weights(C.Structure):
    _fields_ = [("w_router", C.c_void_p), ("router_bias", C.c_void_p),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_down", C.c_void_p),
                ("s_gate", C.c_void_p), ("s_up", C.c_void_p), ("s_down", C.c_void_p),
                ("sh_gate", C.c_void_p), ("sh_up", C.c_void_p), ("sh_down", C.c_void_p),
                ("sh_s_gate", C.c_void_p), ("sh_s_up", C.c_void_p), ("sh_s_down", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = C.CDLL(build())
            L.oracle_f32_to_bf16.restype = C.c_uint16
            L.oracle_f32_to_bf16.argtypes = [C.c_float]
            L.oracle_bf16_round.restype = C.c_float
            L.oracle_bf16_round.argtypes = [C.c_float]
            L.oracle_e4m3_decode.restype = C.c_double
            L.oracle_e4m3_decode.argtypes = [C.c_uint8]
            L.oracle_e4m3_encode.restype = C.c_uint8
            L.oracle_e4m3_encode.argtypes = [C.c_float]
            L.oracle_quantize_row.restype = None
            L.oracle_quantize_row.argtypes = [C.c_void_p, C.c_int, C.c_void_p, C.c_void_p]
            L.oracle_canonical_dot.restype = C.c_float
            L.oracle_canonical_dot.argtypes = [C.c_void_p, C.c_void_p, C.c_int]
            L.oracle_router_logits.restype = None
            L.oracle_router_logits.argtypes = [C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                               C.c_int, C.c_int, C.c_int, C.c_void_p]
            L.oracle_topk.restype = None
            L.oracle_topk.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
            L.oracle_routing_tables.restype = None
            L.oracle_routing_tables.argtypes = [C.c_void_p, C.c_int, C.c_int, C.c_int,
                                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
            L.oracle_moe_forward.restype = C.c_int
            L.oracle_moe_forward.argtypes = [C.POINTER(_Cfg), C.POINTER(_Weights), C.c_void_p,
                                             C.c_void_p, C.c_int, C.c_void_p, C.c_int, C.c_void_p,
                                             C.c_void_p, C.c_void_p, C.c_void_p, C.c_void_p]
            L.oracle_expert_hidden.restype = C.c_int
            L.oracle_expert_hidden.argtypes = [C.POINTER(_Cfg), C.POINTER(_Weights), C.c_void_p, C.c_void_p,
                                               C.c_int, C.c_void_p]
            L.oracle_num_threads.restype = C.c_int
            L.oracle_set_num_threads.restype = None
            L.oracle_set_num_threads.argtypes = [C.c_int]
            _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def _c(a, dtype):
    return None if a is None else np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().oracle_num_threads()


def set_num_threads(n: int) -> None:
    """Thread count of the oracle's parallel loops (timing only)."""
    lib().oracle_set_num_threads(int(n))


# ---------------------------------------------------------------- formats
def bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns, round to nearest even."""
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    return np.array([L.oracle_f32_to_bf16(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def bf16_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def e4m3_decode(codes) -> np.ndarray:
    L = lib()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([L.oracle_e4m3_decode(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    return np.array([L.oracle_e4m3_encode(float(v)) for v in x.ravel()], dtype=np.uint8).reshape(x.shape)


def quantize_rows(x: np.ndarray):
    """Per row, per 128 channels: (codes uint8 [R,C], scales fp32 [R, ceil(C/128)])."""
    L = lib()
    x = _c(x, np.float32)
    R, Cn = x.shape
    q = np.zeros((R, Cn), np.uint8)
    s = np.zeros((R, (Cn + 127) // 128), np.float32)
    for r in range(R):
        L.oracle_quantize_row(_p(x[r]), Cn, _p(q[r]), _p(s[r]))
    return q, s


def canonical_dot(x: np.ndarray, w: np.ndarray) -> np.float32:
    x = _c(x, np.float32)
    w = _c(w, np.float32)
    return np.float32(lib().oracle_canonical_dot(_p(x), _p(w), x.shape[0]))


# ---------------------------------------------------------------- routing
def router_logits(x, w_r, act_dtype: str, bias=None) -> np.ndarray:
    """x [T,H], w_r [H,E] as fp32 arrays (act_dtype 'fp32') or bf16 bits."""
    dt = np.float32 if act_dtype == "fp32" else np.uint16
    x = _c(x, dt)
    w_r = _c(w_r, dt)
    T, H = x.shape
    E = w_r.shape[1]
    out = np.zeros((T, E), np.float32)
    lib().oracle_router_logits(_p(x), _p(w_r), FP32 if act_dtype == "fp32" else BF16,
                               _p(_c(bias, np.float32)), T, H, E, _p(out))
    return out


def topk(logits: np.ndarray, k: int):
    logits = _c(logits, np.float32)
    T, E = logits.shape
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    lib().oracle_topk(_p(logits), T, E, k, _p(idx), _p(w))
    return idx, w


def routing_tables(idx: np.ndarray, E: int):
    idx = _c(idx, np.int32)
    T, k = idx.shape
    counts = np.zeros(E, np.int32)
    offsets = np.zeros(E + 1, np.int32)
    perm = np.zeros(T * k, np.int32)
    pos = np.zeros(T * k, np.int32)
    lib().oracle_routing_tables(_p(idx), T, k, E, _p(counts), _p(offsets), _p(perm), _p(pos))
    return counts, offsets, perm, pos


# ---------------------------------------------------------------- full layer
_WKEYS = ["w_router", "router_bias", "w_gate", "w_up", "w_down", "s_gate", "s_up", "s_down",
          "sh_gate", "sh_up", "sh_down", "sh_s_gate", "sh_s_up", "sh_s_down"]


def _np_weight(key, arr, dtype):
    if arr is None:
        return None
    if key.startswith("s_") or key.startswith("sh_s_") or key == "router_bias":
        return _c(arr, np.float32)
    if key == "w_router":
        return _c(arr, np.float32 if dtype == "fp32" else np.uint16)
    return _c(arr, {"fp32": np.float32, "bf16": np.uint16, "fp8": np.uint8}[dtype])


def moe_forward(cfg: dict, srcs: list, weights: dict, tokens=None):
    """Run the whole layer.

    cfg: dict(H, I, E, k, S, dtype in {'fp32','bf16','fp8'}).
    srcs: list of M arrays [B_m, H] (fp32 or bf16 bits).
    weights: dict with the keys of ``_WKEYS`` (numpy; bf16 as uint16, e4m3 as uint8).
    tokens: optional list of token ids whose outputs to compute.
    Returns dict(out, idx, w, logits, fma) -- out rows follow ``tokens``.
    """
    dtype = cfg["dtype"]
    H, E, k = cfg["H"], cfg["E"], cfg["k"]
    c = _Cfg(H, cfg["I"], E, k, int(cfg.get("S", 0)), DTYPES[dtype])
    keep = {key: _np_weight(key, weights.get(key), dtype) for key in _WKEYS}
    wst = _Weights(*[_p(keep[key]) for key in _WKEYS])
    adt = np.float32 if dtype == "fp32" else np.uint16
    srcs = [_c(s, adt).reshape(-1, H) for s in srcs]
    M = len(srcs)
    counts = np.array([s.shape[0] for s in srcs], dtype=np.int32)
    ptrs = (C.c_void_p * max(M, 1))(*[s.ctypes.data for s in srcs])
    T = int(counts.sum())
    if tokens is None:
        tok = None
        n = T
    else:
        tok = np.ascontiguousarray(np.asarray(tokens, dtype=np.int32))
        n = tok.shape[0]
    out = np.zeros((n, H), np.float32 if dtype == "fp32" else np.uint16)
    idx = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float32)
    logits = np.zeros((T, E), np.float32)
    fma = C.c_longlong(0)
    rc = lib().oracle_moe_forward(C.byref(c), C.byref(wst), C.cast(ptrs, C.c_void_p), _p(counts), M,
                                  _p(tok), n, _p(out), _p(idx), _p(w), _p(logits), C.byref(fma))
    if rc != 0:
        raise ValueError("oracle_moe_forward rejected its arguments")
    return {"out": out, "idx": idx, "w": w, "logits": logits, "fma": int(fma.value)}


def expert_hidden(cfg: dict, weights: dict, x, experts) -> np.ndarray:
    """fp32 SwiGLU hidden rows silu(a Wg) * (a Wu) of (token row, expert) pairs, before
    the down projection's operand rounding (bf16) or quantisation (fp8).

    x: [n, H] token rows (fp32, or bf16 bits for the bf16/fp8 layers); experts: [n]
    expert ids, -1 for the shared expert.  Returns [n, I] fp32."""
    dtype = cfg["dtype"]
    H, I = cfg["H"], cfg["I"]
    c = _Cfg(H, I, cfg["E"], cfg["k"], int(cfg.get("S", 0)), DTYPES[dtype])
    keep = {key: _np_weight(key, weights.get(key), dtype) for key in _WKEYS}
    wst = _Weights(*[_p(keep[key]) for key in _WKEYS])
    x = _c(x, np.float32 if dtype == "fp32" else np.uint16).reshape(-1, H)
    ex = _c(experts, np.int32).reshape(-1)
    if ex.shape[0] != x.shape[0]:
        raise ValueError("one expert id per token row")
    out = np.zeros((x.shape[0], I), np.float32)
    if lib().oracle_expert_hidden(C.byref(c), C.byref(wst), _p(x), _p(ex), x.shape[0], _p(out)) != 0:
        raise ValueError("oracle_expert_hidden rejected an expert id")
    return out
