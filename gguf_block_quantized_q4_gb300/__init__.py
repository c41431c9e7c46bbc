"""Python binding of libmq, the GB300 GGUF block-quantised matmul library.

Argument marshalling only: every step of the computation runs in libmq's CUDA
kernels.  PyTorch provides device memory and streams.  The C ABI
(include/mq.h) is exposed twice:

* ``lib()``: the raw ctypes library with the exact C names and signatures
  (``mq_matvec`` etc.), taking plain pointers and sizes;
* thin wrappers with the same names minus the ``mq_`` prefix that take torch
  tensors, read their data pointers and the current CUDA stream, and raise
  :class:`MQError` on a non-OK status.

There is no fallback: if libmq.so is missing or fails to load, importing the
wrappers raises.
"""
from __future__ import annotations

import ctypes
import os
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libmq.so")

Q4_0, Q4_1, Q5_0, Q5_1, Q8_0, Q4_K, Q5_K, Q6_K = 2, 3, 6, 7, 8, 12, 13, 14
F16, BF16 = 1, 30  # unquantised weights: decode matvec only
REG_DEFAULT, REG_NO_MMQ_PLANE, REG_MMQ_FROM_DECODE_PLANE = 0, 1, 2
# (elements, bytes) per block; f16 / bf16 rows count in units of 32 elements (K % 32 == 0)
BLOCK = {Q4_0: (32, 18), Q4_1: (32, 20), Q5_0: (32, 22), Q5_1: (32, 24), Q8_0: (32, 34),
         Q4_K: (256, 144), Q5_K: (256, 176), Q6_K: (256, 210), F16: (32, 64), BF16: (32, 64)}

STATUS = ["MQ_OK", "MQ_ERR_ARG", "MQ_ERR_TYPE", "MQ_ERR_SHAPE", "MQ_ERR_PAYLOAD",
          "MQ_ERR_ALIGN", "MQ_ERR_CUDA", "MQ_ERR_OOM", "MQ_ERR_LAUNCH", "MQ_ERR_TIMEOUT",
          "MQ_ERR_STATE"]

# The C ABI: name -> (restype, argtypes)
_P, _I64, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
_ST = ctypes.c_int
ABI = {
    "mq_init": (_ST, [ctypes.c_int]),
    "mq_register_weight": (_ST, [ctypes.c_int, _P, _SZ, _I64, _I64, ctypes.c_uint32,
                                 ctypes.POINTER(_P)]),
    "mq_weight_free": (_ST, [_P]),
    "mq_weight_info": (_ST, [_P, ctypes.POINTER(ctypes.c_int), ctypes.POINTER(_I64),
                             ctypes.POINTER(_I64), ctypes.POINTER(_SZ)]),
    "mq_weight_unpack": (_ST, [_P, _P, _SZ]),
    "mq_matvec": (_ST, [ctypes.c_int, _P, _P, _P, _I64, _I64, ctypes.c_int, _P]),
    "mq_act_bytes": (_SZ, [_I64, _I64]),
    "mq_quantize_act": (_ST, [_P, _P, _I64, _I64, _P]),
    "mq_mmq": (_ST, [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mq_mmq_fused": (_ST, [ctypes.c_int, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mq_mmq_fused_static": (_ST, [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mq_matvec_host": (_ST, [ctypes.c_int, _P, _P, _P, _P, _P, _I64, _I64, ctypes.c_int, _P]),
    "mq_mmq_host": (_ST, [ctypes.c_int, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mq_mmq_blockdots": (_ST, [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mq_register_ffn_gu": (_ST, [ctypes.c_int, _P, _P, _SZ, _I64, _I64, ctypes.c_uint32,
                                 ctypes.POINTER(_P)]),
    "mq_ffn_gu_matvec": (_ST, [ctypes.c_int, _P, _P, _P, _I64, _I64, ctypes.c_int, _P]),
    "mq_ffn_gu_mmq": (_ST, [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _P]),
    "mq_stream_status": (_ST, [_P]),
    "mq_last_error": (ctypes.c_char_p, []),
    "mq_status_name": (ctypes.c_char_p, [ctypes.c_int]),
}

_lib = None


class MQError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS[status] if 0 <= status < len(STATUS) else f"status {status}"
        super().__init__(f"{self.name}: {message}")


def lib():
    """Load libmq.so (built in-tree by build.py) and declare the C ABI."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: build it with "
                              "`python -m gguf_block_quantized_q4_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in ABI.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(status: int):
    if status != 0:
        raise MQError(status, lib().mq_last_error().decode(errors="replace"))


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def init(device: int = 0):
    _check(lib().mq_init(device))


class Weight:
    """A registered weight (library-owned device planes)."""

    def __init__(self, qtype: int, data, N: int, K: int, flags: int = REG_DEFAULT):
        import numpy as np
        buf = np.ascontiguousarray(np.frombuffer(memoryview(data), dtype=np.uint8)
                                   if not isinstance(data, np.ndarray) else data.view(np.uint8))
        h = ctypes.c_void_p()
        _check(lib().mq_register_weight(qtype, buf.ctypes.data_as(ctypes.c_void_p), buf.nbytes,
                                        N, K, flags, ctypes.byref(h)))
        self.handle = h
        self.qtype, self.N, self.K = qtype, N, K
        self.nbytes = buf.nbytes

    def info(self):
        t, n, k, b = ctypes.c_int(), _I64(), _I64(), _SZ()
        _check(lib().mq_weight_info(self.handle, ctypes.byref(t), ctypes.byref(n),
                                    ctypes.byref(k), ctypes.byref(b)))
        return t.value, n.value, k.value, b.value

    def unpack(self):
        import numpy as np
        out = np.empty(self.nbytes, dtype=np.uint8)
        _check(lib().mq_weight_unpack(self.handle, out.ctypes.data_as(ctypes.c_void_p),
                                      out.nbytes))
        return out

    def free(self):
        if self.handle:
            _free_deferred()
            _check(lib().mq_weight_free(self.handle))
            self.handle = None

    def __del__(self):
        # mq_weight_free synchronises the device, which would invalidate a stream capture in
        # progress (a weight kept alive by a reference cycle is collected whenever the
        # garbage collector runs): during a capture the handle is kept and freed later
        try:
            if getattr(self, "handle", None) and _lib is not None:
                if _capturing():
                    _deferred_frees.append(self.handle)
                else:
                    _free_deferred()
                    _lib.mq_weight_free(self.handle)
        except Exception:
            pass


_deferred_frees = []


def _capturing() -> bool:
    torch = sys.modules.get("torch")
    try:
        return bool(torch is not None and torch.cuda.is_available()
                    and torch.cuda.is_current_stream_capturing())
    except Exception:
        return False


def _free_deferred():
    """Free the weights whose collection fell inside a stream capture (none while one is
    still in progress)."""
    if not _deferred_frees or _capturing():
        return
    while _deferred_frees:
        _lib.mq_weight_free(_deferred_frees.pop())


def register_weight(qtype, data, N, K, flags=REG_DEFAULT) -> Weight:
    _free_deferred()
    return Weight(qtype, data, N, K, flags)


class FfnGuWeight(Weight):
    """A fused gate/up weight (mq_register_ffn_gu): N gate rows and N up rows."""

    def __init__(self, qtype: int, gate, up, N: int, K: int, flags: int = REG_DEFAULT):
        import numpy as np

        def as_u8(d):
            return np.ascontiguousarray(np.frombuffer(memoryview(d), dtype=np.uint8)
                                        if not isinstance(d, np.ndarray) else d.view(np.uint8))
        g, u = as_u8(gate), as_u8(up)
        if g.nbytes != u.nbytes:
            raise ValueError("gate and up payloads differ in size")
        h = ctypes.c_void_p()
        _check(lib().mq_register_ffn_gu(qtype, g.ctypes.data_as(ctypes.c_void_p),
                                        u.ctypes.data_as(ctypes.c_void_p), g.nbytes, N, K, flags,
                                        ctypes.byref(h)))
        self.handle = h
        self.qtype, self.N, self.K = qtype, N, K
        self.nbytes = 2 * g.nbytes


def register_ffn_gu(qtype, gate, up, N, K, flags=REG_DEFAULT) -> FfnGuWeight:
    _free_deferred()
    return FfnGuWeight(qtype, gate, up, N, K, flags)


def ffn_gu_matvec(W: FfnGuWeight, x, h=None, stream=None):
    """h[B][N] = silu(W_gate x) * (W_up x) (x: CUDA f32 [B][K] or [K])."""
    import torch
    x2 = x.reshape(-1, W.K)
    B = x2.shape[0]
    if h is None:
        h = torch.empty((B, W.N), dtype=torch.float32, device=x.device)
    _check(lib().mq_ffn_gu_matvec(W.qtype, W.handle, _ptr(x2), _ptr(h), W.N, W.K, B,
                                  _stream(stream)))
    return h


def ffn_gu_mmq(W: FfnGuWeight, xq, M: int, h=None, stream=None):
    """h[M][N] = silu(W_gate a) * (W_up a) for the quantised activations xq."""
    import torch
    if h is None:
        h = torch.empty((M, W.N), dtype=torch.float32, device=xq.device)
    _check(lib().mq_ffn_gu_mmq(W.qtype, W.handle, _ptr(xq), _ptr(h), M, W.N, W.K,
                               _stream(stream)))
    return h


def matvec(W: Weight, x, y=None, stream=None):
    """y[B][N] = dequant(W) @ x[B][K]^T (x: CUDA f32 [B][K] or [K])."""
    import torch
    x2 = x.reshape(-1, W.K)
    B = x2.shape[0]
    if y is None:
        y = torch.empty((B, W.N), dtype=torch.float32, device=x.device)
    _check(lib().mq_matvec(W.qtype, W.handle, _ptr(x2), _ptr(y), W.N, W.K, B, _stream(stream)))
    return y


def act_bytes(M: int, K: int) -> int:
    return lib().mq_act_bytes(M, K)


def min_ld(nb: int) -> int:
    """Row stride (f16 elements) of the min-term operand: 3*nb rounded up to 8."""
    return (3 * nb + 7) // 8 * 8


def act_layout(M: int, K: int):
    """Byte offsets of the xq sections (see mq_act_bytes in mq.h)."""
    def al(v):
        return (v + 255) & ~255
    mt = (M + 127) // 128 * 128
    nb = K // 32
    o = {"qs": 0}
    o["scale"] = al(o["qs"] + M * K)
    o["bsum"] = al(o["scale"] + M * nb * 4)
    o["op"] = al(o["bsum"] + M * nb * 4)
    o["scaleT"] = al(o["op"] + M * K * 2)
    o["minT"] = al(o["scaleT"] + mt * nb * 4)
    o["amin"] = al(o["minT"] + mt * nb * 4)
    o["urow"] = al(o["amin"] + M * min_ld(nb) * 2)
    o["sync"] = al(o["urow"] + mt * 4)
    o["total"] = al(o["sync"] + 8)
    o["mt"] = mt
    return o


def act_views(xq, M: int, K: int):
    """Views (qs int8 [M][K], scale f32 [M][K/32], bsum int32 [M][K/32], op f16 [M][K])
    of an xq buffer, following the layout documented in mq.h."""
    import torch
    o = act_layout(M, K)
    nb = K // 32
    qs = xq[o["qs"]:o["qs"] + M * K].view(torch.int8).view(M, K)
    sc = xq[o["scale"]:o["scale"] + M * nb * 4].view(torch.float32).view(M, nb)
    bs = xq[o["bsum"]:o["bsum"] + M * nb * 4].view(torch.int32).view(M, nb)
    op = xq[o["op"]:o["op"] + M * K * 2].view(torch.float16).view(M, K)
    return qs, sc, bs, op


def act_views_transposed(xq, M: int, K: int):
    """Views (scaleT f32 [K/32][M], minT f32 [K/32][M]) of the transposed sections."""
    import torch
    o = act_layout(M, K)
    nb, mt = K // 32, o["mt"]
    st = xq[o["scaleT"]:o["scaleT"] + mt * nb * 4].view(torch.float32).view(nb, mt)[:, :M]
    tt = xq[o["minT"]:o["minT"] + mt * nb * 4].view(torch.float32).view(nb, mt)[:, :M]
    return st, tt


def act_views_min(xq, M: int, K: int):
    """Views (amin f16 [M][3*K/32], urow f32 [M]) of the min-term operand sections."""
    import torch
    o = act_layout(M, K)
    nb = K // 32
    ld = min_ld(nb)
    am = xq[o["amin"]:o["amin"] + M * ld * 2].view(torch.float16).view(M, ld)[:, :3 * nb]
    ur = xq[o["urow"]:o["urow"] + M * 4].view(torch.float32)
    return am, ur


def quantize_act(x, xq=None, stream=None):
    """Quantise CUDA f32 x[M][K]; returns the uint8 xq buffer."""
    import torch
    M, K = x.shape
    if xq is None:
        xq = torch.empty(act_bytes(M, K), dtype=torch.uint8, device=x.device)
    _check(lib().mq_quantize_act(_ptr(x), _ptr(xq), M, K, _stream(stream)))
    return xq


def mmq(W: Weight, xq, M: int, y=None, stream=None):
    import torch
    if y is None:
        y = torch.empty((M, W.N), dtype=torch.float32, device=xq.device)
    _check(lib().mq_mmq(W.qtype, W.handle, _ptr(xq), _ptr(y), M, W.N, W.K, _stream(stream)))
    return y


def act_buffer(M: int, K: int, device=None):
    """An xq buffer of mq_act_bytes(M, K) bytes, zero-filled (so the fused call's barrier
    count starts at zero), ready for mmq_fused as well as quantize_act."""
    import torch
    return torch.zeros(act_bytes(M, K), dtype=torch.uint8, device=device or "cuda")


def mmq_fused(W: Weight, x, xq=None, y=None, stream=None):
    """Quantise x (f32 [M][K] on the device) into xq and run the MMQ, in one kernel.
    Returns (y, xq); xq then holds what quantize_act writes."""
    import torch
    M = x.shape[0]
    if xq is None:
        xq = act_buffer(M, W.K, x.device)
    if y is None:
        y = torch.empty((M, W.N), dtype=torch.float32, device=x.device)
    _check(lib().mq_mmq_fused(W.qtype, W.handle, _ptr(x), _ptr(xq), _ptr(y), M, W.N, W.K,
                              _stream(stream)))
    return y, xq


def matvec_host(W: Weight, x_host, y_host, x_dev, y_dev, stream=None):
    """Decode matvec from host buffers (torch CPU tensors x_host [B][K], y_host [B][N]), all
    enqueued on the stream by one C call.  Pinned, 16-byte aligned host tensors are read and
    written by the kernels directly (x through x_dev, y straight into y_host); others are
    copied through x_dev / y_dev.  y_host is complete when the stream is."""
    B = x_host.shape[0]
    _check(lib().mq_matvec_host(W.qtype, W.handle, _ptr(x_host), _ptr(y_host), _ptr(x_dev),
                                _ptr(y_dev), W.N, W.K, B, _stream(stream)))


def mmq_host(W: Weight, x_host, y_host, x_dev, xq_dev, y_dev, stream=None):
    """Prefill (quantise + MMQ) from host buffers, as matvec_host: a pinned, 16-byte aligned
    x_host is read by the quantiser directly (else copied through x_dev); y goes out through
    y_dev and a copy."""
    M = x_host.shape[0]
    _check(lib().mq_mmq_host(W.qtype, W.handle, _ptr(x_host), _ptr(y_host), _ptr(x_dev),
                             _ptr(xq_dev), _ptr(y_dev), M, W.N, W.K, _stream(stream)))


STATIC_XQ_BYTES = 16 << 20  # the library's scratch for mmq_fused_static (MQ_STATIC_XQ_BYTES)


def mmq_fused_static(W: Weight, x, y=None, stream=None):
    """mmq_fused with the library's static scratch in place of an xq buffer (allocates
    nothing on the device; one call in flight at a time).  Returns y."""
    import torch
    M = x.shape[0]
    if y is None:
        y = torch.empty((M, W.N), dtype=torch.float32, device=x.device)
    _check(lib().mq_mmq_fused_static(W.qtype, W.handle, _ptr(x), _ptr(y), M, W.N, W.K,
                                     _stream(stream)))
    return y


def mmq_blockdots(W: Weight, xq, M: int, D=None, stream=None):
    import torch
    if D is None:
        D = torch.empty((M, W.N, W.K // 32), dtype=torch.int32, device=xq.device)
    _check(lib().mq_mmq_blockdots(W.qtype, W.handle, _ptr(xq), _ptr(D), M, W.N, W.K,
                                  _stream(stream)))
    return D


def stream_status(stream=None):
    _check(lib().mq_stream_status(_stream(stream)))
