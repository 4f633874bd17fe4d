"""Thin Python binding of libafd_ffn.so (include/afd_ffn.h).

Argument marshalling only: every step of the layer runs in the library's CUDA
kernels.  The same names as the C ABI are exported (``afd_ffn_create``,
``afd_ffn_forward``, ...); ``MoELayer`` wraps them for torch tensors.  If the
shared library has not been built, loading raises -- there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libafd_ffn.so")

AFD_FP32, AFD_BF16, AFD_FP8_E4M3 = 0, 1, 2
DTYPE_CODES = {"fp32": AFD_FP32, "bf16": AFD_BF16, "fp8": AFD_FP8_E4M3}
AFD_OK, AFD_EINVAL, AFD_ECUDA, AFD_ECAPACITY, AFD_EUNSUPPORTED, AFD_EDEVICE = 0, -1, -2, -3, -4, -5
AFD_MAX_SOURCES, AFD_MAX_MICRO = 64, 4

AFD_NUM_KERNELS = 6
INJECT_TIMEOUT = 1
INJECT_RANGE = 2
KERNEL_NAMES = ["router", "routing", "pack", "gemm_gateup", "gemm_down", "combine"]

EXPORTS = ["afd_ffn_create", "afd_ffn_create_error", "afd_ffn_forward", "afd_ffn_forward_pipelined",
           "afd_ffn_forward_host", "afd_ffn_forward_host_async", "afd_ffn_host_wait", "afd_ffn_debug_routing",
           "afd_ffn_debug_operands", "afd_ffn_debug_inject", "afd_ffn_check", "afd_ffn_last_error",
           "afd_ffn_profile_begin", "afd_ffn_profile_end", "afd_ffn_launches_per_forward",
           "afd_ffn_device_bytes", "afd_ffn_router_noalloc", "afd_ffn_destroy"]


class AfdConfig(C.Structure):
    _fields_ = [("H", C.c_int), ("I", C.c_int), ("E", C.c_int), ("k", C.c_int), ("n_shared", C.c_int),
                ("max_sources", C.c_int), ("max_tokens", C.c_int), ("dtype", C.c_int)]


class AfdWeights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w_router", "router_bias", "w_gate", "w_up", "w_down", "s_gate", "s_up",
                                          "s_down", "sh_gate", "sh_up", "sh_down", "sh_s_gate", "sh_s_up",
                                          "sh_s_down")]


class AfdError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"afd_ffn error {code}: {msg}")
        self.code = code


_lib = None


def lib():
    """Load libafd_ffn.so (raises if it is missing)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built: run __graft_entry__.build() first")
        L = C.CDLL(LIB_PATH)
        vp, ip = C.c_void_p, C.c_int
        L.afd_ffn_create.argtypes = [C.POINTER(AfdConfig), C.POINTER(AfdWeights), C.POINTER(vp)]
        L.afd_ffn_create.restype = ip
        L.afd_ffn_create_error.restype = C.c_char_p
        L.afd_ffn_forward.argtypes = [vp, vp, vp, vp, ip, vp]
        L.afd_ffn_forward.restype = ip
        L.afd_ffn_forward_pipelined.argtypes = [vp, vp, ip, vp, vp, ip, vp]
        L.afd_ffn_forward_pipelined.restype = ip
        L.afd_ffn_forward_host.argtypes = [vp, vp, ip, vp, vp, ip, vp]
        L.afd_ffn_forward_host.restype = ip
        L.afd_ffn_forward_host_async.argtypes = [vp, ip, vp, vp, ip, vp]
        L.afd_ffn_forward_host_async.restype = ip
        L.afd_ffn_host_wait.argtypes = [vp]
        L.afd_ffn_host_wait.restype = ip
        L.afd_ffn_debug_inject.argtypes = [vp, vp, ip, C.c_longlong]
        L.afd_ffn_debug_inject.restype = ip
        L.afd_ffn_debug_routing.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp]
        L.afd_ffn_debug_routing.restype = ip
        L.afd_ffn_debug_operands.argtypes = [vp, vp, vp, vp, vp, vp]
        L.afd_ffn_debug_operands.restype = ip
        L.afd_ffn_check.argtypes = [vp, vp]
        L.afd_ffn_check.restype = ip
        L.afd_ffn_last_error.argtypes = [vp]
        L.afd_ffn_last_error.restype = C.c_char_p
        L.afd_ffn_profile_begin.argtypes = [vp]
        L.afd_ffn_profile_begin.restype = ip
        L.afd_ffn_profile_end.argtypes = [vp, vp, vp]
        L.afd_ffn_profile_end.restype = ip
        L.afd_ffn_launches_per_forward.argtypes = [vp, ip]
        L.afd_ffn_launches_per_forward.restype = ip
        L.afd_ffn_device_bytes.argtypes = [vp]
        L.afd_ffn_device_bytes.restype = C.c_size_t
        L.afd_ffn_router_noalloc.argtypes = [vp, vp, vp, ip, ip, ip, ip, ip, vp, vp, vp, vp]
        L.afd_ffn_router_noalloc.restype = ip
        L.afd_ffn_destroy.argtypes = [vp]
        L.afd_ffn_destroy.restype = None
        _lib = L
    return _lib


def _ptr_array(ptrs):
    n = max(len(ptrs), 1)
    return (C.c_void_p * n)(*[p if p else None for p in ptrs])


def _int_array(vals):
    n = max(len(vals), 1)
    return (C.c_int * n)(*vals)


def _check(rc, handle=None):
    if rc != AFD_OK:
        msg = (lib().afd_ffn_last_error(handle) if handle else lib().afd_ffn_create_error()) or b""
        raise AfdError(rc, msg.decode())
    return rc


# ------------------------------------------------------------ C ABI, same names
def afd_ffn_create(cfg: AfdConfig, weights: AfdWeights):
    h = C.c_void_p()
    _check(lib().afd_ffn_create(C.byref(cfg), C.byref(weights), C.byref(h)))
    return h


def afd_ffn_forward(h, stream, src_ptrs, src_counts, out_ptrs):
    return _check(lib().afd_ffn_forward(h, stream, _ptr_array(src_ptrs), _int_array(src_counts), len(src_counts),
                                        _ptr_array(out_ptrs)), h)


def afd_ffn_forward_pipelined(h, stream, n_micro, src_ptrs, src_counts, out_ptrs):
    return _check(lib().afd_ffn_forward_pipelined(h, stream, n_micro, _ptr_array(src_ptrs), _int_array(src_counts),
                                                  len(src_counts), _ptr_array(out_ptrs)), h)


def afd_ffn_forward_host(h, stream, n_micro, src_ptrs, src_counts, out_ptrs):
    return _check(lib().afd_ffn_forward_host(h, stream, n_micro, _ptr_array(src_ptrs), _int_array(src_counts),
                                             len(src_counts), _ptr_array(out_ptrs)), h)


def afd_ffn_forward_host_async(h, n_micro, src_ptrs, src_counts, out_ptrs):
    return _check(lib().afd_ffn_forward_host_async(h, n_micro, _ptr_array(src_ptrs), _int_array(src_counts),
                                                   len(src_counts), _ptr_array(out_ptrs)), h)


def afd_ffn_host_wait(h):
    return _check(lib().afd_ffn_host_wait(h), h)


def afd_ffn_debug_inject(h, stream, kind, arg):
    return _check(lib().afd_ffn_debug_inject(h, stream, kind, arg), h)


def afd_ffn_debug_routing(h, stream, topk_idx, topk_w, counts, offsets, perm_token, pos, logits):
    return _check(lib().afd_ffn_debug_routing(h, stream, topk_idx, topk_w, counts, offsets, perm_token, pos,
                                              logits), h)


def afd_ffn_debug_operands(h, stream, P, P_scale, Hmid, H_scale):
    return _check(lib().afd_ffn_debug_operands(h, stream, P, P_scale, Hmid, H_scale), h)


def afd_ffn_check(h, stream):
    return _check(lib().afd_ffn_check(h, stream), h)


def afd_ffn_last_error(h) -> str:
    return (lib().afd_ffn_last_error(h) or b"").decode()


def afd_ffn_profile_begin(h):
    return _check(lib().afd_ffn_profile_begin(h), h)


def afd_ffn_profile_end(h):
    """-> (list of summed ms per kernel, number of recorded forwards)"""
    ms = (C.c_double * AFD_NUM_KERNELS)()
    n = C.c_int(0)
    _check(lib().afd_ffn_profile_end(h, ms, C.byref(n)), h)
    return list(ms), n.value


def afd_ffn_launches_per_forward(h, T) -> int:
    n = int(lib().afd_ffn_launches_per_forward(h, int(T)))
    if n < 0:
        raise AfdError(n, "launches_per_forward: bad handle or T")
    return n


def afd_ffn_device_bytes(h) -> int:
    return int(lib().afd_ffn_device_bytes(h))


def afd_ffn_router_noalloc(stream, src_ptrs, src_counts, H, E, k, dtype, w_router, router_bias, topk_idx,
                           topk_w) -> int:
    """Routing (top-k indices and weights) with no device allocation; returns
    the status code (0 = ok).  Pointers are device addresses (ints)."""
    return int(lib().afd_ffn_router_noalloc(stream, _ptr_array(src_ptrs), _int_array(src_counts), len(src_counts),
                                            H, E, k, DTYPE_CODES[dtype] if isinstance(dtype, str) else dtype,
                                            w_router, router_bias, topk_idx, topk_w))


def afd_ffn_destroy(h):
    lib().afd_ffn_destroy(h)


# ------------------------------------------------------------ torch convenience
class MoELayer:
    """One FFN-server MoE layer on the current CUDA device.

    ``weights``: dict of CUDA tensors in the layer's input format (keys as in
    ``synth.make_weights``).  The library copies them at construction."""

    def __init__(self, H, I, E, k, dtype, weights, n_shared=0, max_tokens=4096, max_sources=16):
        import torch

        self.torch = torch
        self.H, self.I, self.E, self.k, self.S = H, I, E, k, n_shared
        self.dtype = dtype
        self.act_dtype = torch.float32 if dtype == "fp32" else torch.bfloat16
        self.max_tokens = max_tokens
        cfg = AfdConfig(H, I, E, k, n_shared, max_sources, max_tokens, DTYPE_CODES[dtype])
        w = AfdWeights()
        for name, _ in AfdWeights._fields_:
            t = weights.get(name)
            if t is not None:
                assert t.is_cuda and t.is_contiguous(), name
                setattr(w, name, t.data_ptr())
        self.handle = afd_ffn_create(cfg, w)

    def close(self):
        if getattr(self, "handle", None):
            afd_ffn_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def _stream(self, stream):
        s = stream if stream is not None else self.torch.cuda.current_stream()
        return C.c_void_p(s.cuda_stream)

    def new_outputs(self, srcs):
        return [self.torch.empty_like(s) for s in srcs]

    def forward(self, srcs, outs=None, stream=None, n_micro=1):
        outs = self.new_outputs(srcs) if outs is None else outs
        sp = [s.data_ptr() if s.shape[0] else 0 for s in srcs]
        op = [o.data_ptr() if o.shape[0] else 0 for o in outs]
        counts = [int(s.shape[0]) for s in srcs]
        if n_micro == 1:
            afd_ffn_forward(self.handle, self._stream(stream), sp, counts, op)
        else:
            afd_ffn_forward_pipelined(self.handle, self._stream(stream), n_micro, sp, counts, op)
        return outs

    def forward_host(self, srcs, outs, stream=None, n_micro=1):
        """Host tensors in and out (pinned for asynchronous copies); synchronous.
        n_micro > 1 runs the micro-batch pipeline between the copies."""
        sp = [s.data_ptr() if s.shape[0] else 0 for s in srcs]
        op = [o.data_ptr() if o.shape[0] else 0 for o in outs]
        afd_ffn_forward_host(self.handle, self._stream(stream), int(n_micro), sp, [int(s.shape[0]) for s in srcs],
                             op)
        return outs

    def forward_host_async(self, srcs, outs, n_micro=1):
        """Host tensors in and out (pinned), asynchronous: returns once the copies and the
        layer are enqueued on the library's streams; consecutive calls overlap one batch's
        transfers with another's compute.  Outputs are valid after host_wait()."""
        sp = [s.data_ptr() if s.shape[0] else 0 for s in srcs]
        op = [o.data_ptr() if o.shape[0] else 0 for o in outs]
        afd_ffn_forward_host_async(self.handle, int(n_micro), sp, [int(s.shape[0]) for s in srcs], op)
        return outs

    def host_wait(self):
        """Wait for every forward_host_async call so far."""
        return afd_ffn_host_wait(self.handle)

    def routing(self, T, stream=None):
        """Routing tables of the last forward (of its first micro-batch when it was
        micro-batched) as int32/fp32 tensors."""
        torch = self.torch
        dev = torch.device("cuda")
        r = {
            "idx": torch.empty(T * self.k, dtype=torch.int32, device=dev),
            "w": torch.empty(T * self.k, dtype=torch.float32, device=dev),
            "counts": torch.empty(self.E, dtype=torch.int32, device=dev),
            "offsets": torch.empty(self.E + 1, dtype=torch.int32, device=dev),
            "perm": torch.empty(T * self.k, dtype=torch.int32, device=dev),
            "pos": torch.empty(T * self.k, dtype=torch.int32, device=dev),
            "logits": torch.empty(T * self.E, dtype=torch.float32, device=dev),
        }
        afd_ffn_debug_routing(self.handle, self._stream(stream), *[r[k].data_ptr() for k in
                                                                   ("idx", "w", "counts", "offsets", "perm", "pos",
                                                                    "logits")])
        return r

    def operands(self, T, stream=None, with_P=True):
        """Expert-GEMM operands of the last forward (of its first micro-batch when it was
        micro-batched): packed token rows P [R, H] and SwiGLU rows h [R, I], R = T*(k+S),
        in the layer's operand format (uint8 e4m3 codes for fp8, with scales
        [H/128, R] and [I/128, R]).  with_P=False skips P (a bf16 forward of at most 8
        tokens writes none, and the library rejects the request)."""
        torch = self.torch
        dev = torch.device("cuda")
        R = T * (self.k + self.S)
        et = {"fp32": torch.float32, "bf16": torch.bfloat16, "fp8": torch.uint8}[self.dtype]
        r = {"h": torch.empty(R, self.I, dtype=et, device=dev)}
        if with_P:
            r["P"] = torch.empty(R, self.H, dtype=et, device=dev)
        if self.dtype == "fp8":
            r["P_scale"] = torch.empty(self.H // 128, R, dtype=torch.float32, device=dev)
            r["h_scale"] = torch.empty(self.I // 128, R, dtype=torch.float32, device=dev)
        afd_ffn_debug_operands(self.handle, self._stream(stream), r["P"].data_ptr() if with_P else None,
                               r["P_scale"].data_ptr() if "P_scale" in r else None, r["h"].data_ptr(),
                               r["h_scale"].data_ptr() if "h_scale" in r else None)
        return r

    def debug_inject(self, kind, arg=0, stream=None):
        """Make a device-side check fire (INJECT_TIMEOUT: a bounded wait that runs out after
        ``arg`` cycles; INJECT_RANGE: an out-of-range expert id in the routing tables); the
        next check() reports it."""
        return afd_ffn_debug_inject(self.handle, self._stream(stream), int(kind), int(arg))

    def check(self, stream=None):
        return afd_ffn_check(self.handle, self._stream(stream))

    def profile_begin(self):
        afd_ffn_profile_begin(self.handle)

    def profile_end(self):
        """-> (dict kernel name -> summed ms, number of recorded forwards)"""
        ms, n = afd_ffn_profile_end(self.handle)
        return dict(zip(KERNEL_NAMES, ms)), n

    def launches_per_forward(self, T):
        """Kernel launches one forward of T tokens enqueues."""
        return afd_ffn_launches_per_forward(self.handle, T)

    @property
    def device_bytes(self):
        return afd_ffn_device_bytes(self.handle)
