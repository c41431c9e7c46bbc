"""Python access to the CPU oracle (oracle.c) for the tests, the smoke check and
the bench's CPU-baseline leg.

TEST INFRASTRUCTURE ONLY: the product package never imports this module.  It
shares no code with the CUDA library; the only code the two sides share is the
seeded input generator module ``synth``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_LIB_OMP = os.path.join(_HERE, "liboracle_omp.so")

CFLAGS = ["-std=c99", "-O2", "-fno-fast-math", "-ffp-contract=off", "-Wall",
          "-Wno-unknown-pragmas", "-shared", "-fPIC"]


def _compile(target: str, extra, force: bool) -> str:
    if force or not os.path.exists(target) or \
            os.path.getmtime(target) < os.path.getmtime(_SRC):
        tmp = target + f".tmp{os.getpid()}"
        subprocess.run(["gcc", *CFLAGS, *extra, _SRC, "-o", tmp, "-lm"], check=True,
                       capture_output=True)
        os.replace(tmp, target)
    return target


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no FMA contraction), and the
    same source with -fopenmp into liboracle_omp.so when the compiler has OpenMP (the
    all-cores build: rows in parallel, each row's arithmetic unchanged)."""
    lib_path = _compile(_LIB, [], force)
    try:
        _compile(_LIB_OMP, ["-fopenmp"], force)
    except (subprocess.CalledProcessError, OSError):
        pass  # no OpenMP here: the all-cores build is absent, lib_omp() returns None
    return lib_path


_lib = None
_lib_omp = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64


def load(path: str):
    """A ctypes handle on a compiled oracle library, its signatures declared."""
    L = ctypes.CDLL(path)
    L.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_f16_to_double.restype = ctypes.c_double
    L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    L.oracle_bf16_to_double.restype = ctypes.c_double
    L.oracle_q4_k_scale_min.argtypes = [_P, ctypes.c_int, _P, _P]
    L.oracle_q4_k_scale_min.restype = None
    L.oracle_dequant_row.argtypes = [ctypes.c_int, _P, _I64, _P]
    L.oracle_int_weights_row.argtypes = [ctypes.c_int, _P, _I64, _P]
    L.oracle_matvec.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, ctypes.c_int, _I64, _I64,
                                _P, _P]
    L.oracle_quantize_act.argtypes = [_P, _I64, _I64, _P, _P, _P]
    L.oracle_blockdots.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, _I64, _P, _I64, _I64,
                                   _I64, _P]
    L.oracle_mmq.argtypes = [ctypes.c_int, _P, _I64, _I64, _P, _P, _I64, _P, _I64, _I64,
                             _I64, _P, _P]
    for f in ("oracle_dequant_row", "oracle_int_weights_row", "oracle_matvec",
              "oracle_quantize_act", "oracle_blockdots", "oracle_mmq"):
        getattr(L, f).restype = ctypes.c_int
    L.oracle_threads.argtypes = []
    L.oracle_threads.restype = ctypes.c_int
    L.oracle_set_threads.argtypes = [ctypes.c_int]
    L.oracle_set_threads.restype = None
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(build())
    return _lib


def lib_omp():
    """The OpenMP build of the same oracle.c (rows over all cores), or None if this host's
    compiler has no OpenMP."""
    global _lib_omp
    if _lib_omp is None:
        build()
        if os.path.exists(_LIB_OMP):
            _lib_omp = load(_LIB_OMP)
    return _lib_omp


def threads(parallel: bool = True) -> int:
    """Threads the row loops run on: 1 for the plain build, the OpenMP build's count else."""
    L = lib_omp() if parallel else lib()
    return L.oracle_threads() if L is not None else 1


def _rows_lib(parallel: bool):
    if parallel:
        L = lib_omp()
        if L is not None:
            return L
    return lib()


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} failed (rc={rc})")


def f16_to_double(bits: int) -> float:
    return lib().oracle_f16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return lib().oracle_bf16_to_double(bits)


def q4_k_scale_min(s12: bytes, j: int):
    buf = np.frombuffer(bytes(s12), dtype=np.uint8).copy()
    sc, mn = ctypes.c_int(), ctypes.c_int()
    lib().oracle_q4_k_scale_min(_ptr(buf), j, ctypes.byref(sc), ctypes.byref(mn))
    return sc.value, mn.value


def dequant_row(qtype: int, row: np.ndarray, K: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    out = np.empty(K, dtype=np.float64)
    _check(lib().oracle_dequant_row(qtype, _ptr(row), K, _ptr(out)), "dequant_row")
    return out


def dequant(qtype: int, W: np.ndarray, N: int, K: int) -> np.ndarray:
    W = np.ascontiguousarray(W, dtype=np.uint8).reshape(N, -1)
    return np.stack([dequant_row(qtype, W[n], K) for n in range(N)]) if N else \
        np.zeros((0, K))


def int_weights_row(qtype: int, row: np.ndarray, K: int) -> np.ndarray:
    row = np.ascontiguousarray(row, dtype=np.uint8)
    out = np.empty(K, dtype=np.int64)
    _check(lib().oracle_int_weights_row(qtype, _ptr(row), K, _ptr(out)), "int_weights_row")
    return out


def matvec(qtype: int, W: np.ndarray, N: int, K: int, x: np.ndarray, n0: int = 0,
           n1: int | None = None, parallel: bool = False):
    """Returns (y, bound), each float64 [B][n1-n0].  parallel: rows on all cores (the
    OpenMP build of the same source; the same bits)."""
    n1 = N if n1 is None else n1
    x = np.ascontiguousarray(x, dtype=np.float32).reshape(-1, K)
    B = x.shape[0]
    W = np.ascontiguousarray(W, dtype=np.uint8)
    y = np.empty((B, n1 - n0), dtype=np.float64)
    bnd = np.empty_like(y)
    _check(_rows_lib(parallel).oracle_matvec(qtype, _ptr(W), N, K, _ptr(x), B, n0, n1, _ptr(y),
                                             _ptr(bnd)), "matvec")
    return y, bnd


def quantize_act(x: np.ndarray):
    """Returns (qs int8 [M][K], scale f32 [M][K/32], bsum int32 [M][K/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    M, K = x.shape
    qs = np.empty((M, K), dtype=np.int8)
    sc = np.empty((M, K // 32), dtype=np.float32)
    bs = np.empty((M, K // 32), dtype=np.int32)
    _check(lib().oracle_quantize_act(_ptr(x), M, K, _ptr(qs), _ptr(sc), _ptr(bs)),
           "quantize_act")
    return qs, sc, bs


def blockdots(qtype: int, W: np.ndarray, N: int, K: int, qs: np.ndarray, mrows=None,
              n0: int = 0, n1: int | None = None, parallel: bool = False) -> np.ndarray:
    """Returns int64 D [len(mrows)][n1-n0][K/32]."""
    n1 = N if n1 is None else n1
    qs = np.ascontiguousarray(qs, dtype=np.int8)
    M = qs.shape[0]
    mrows = np.arange(M, dtype=np.int64) if mrows is None else \
        np.ascontiguousarray(mrows, dtype=np.int64)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    D = np.empty((len(mrows), n1 - n0, K // 32), dtype=np.int64)
    _check(_rows_lib(parallel).oracle_blockdots(qtype, _ptr(W), N, K, _ptr(qs), M, _ptr(mrows),
                                                len(mrows), n0, n1, _ptr(D)), "blockdots")
    return D


def mmq(qtype: int, W: np.ndarray, N: int, K: int, qs: np.ndarray, scale: np.ndarray,
        mrows=None, n0: int = 0, n1: int | None = None, parallel: bool = False):
    """Returns (y, bound), float64 [len(mrows)][n1-n0]."""
    n1 = N if n1 is None else n1
    qs = np.ascontiguousarray(qs, dtype=np.int8)
    scale = np.ascontiguousarray(scale, dtype=np.float32)
    M = qs.shape[0]
    mrows = np.arange(M, dtype=np.int64) if mrows is None else \
        np.ascontiguousarray(mrows, dtype=np.int64)
    W = np.ascontiguousarray(W, dtype=np.uint8)
    y = np.empty((len(mrows), n1 - n0), dtype=np.float64)
    bnd = np.empty_like(y)
    _check(_rows_lib(parallel).oracle_mmq(qtype, _ptr(W), N, K, _ptr(qs), _ptr(scale), M,
                                          _ptr(mrows), len(mrows), n0, n1, _ptr(y), _ptr(bnd)),
           "mmq")
    return y, bnd


# ---- fused FFN gate/up with SwiGLU ("minfer CUDA Backend Design" §4.3 FusedFFN and
# SwiGLU ops, §4.6 the ffn_gu concat of the gate and up weights).  The pages name the
# operation but do not write it out; the reading used here is the usual one,
# h = silu(g) * u with silu(v) = v / (1 + exp(-v)), g = W_gate x, u = W_up x.

SILU_SLOPE = 1.1  # max |silu'(v)| = 1.0998... (at v ~ 2.4), rounded up


def silu(v) -> np.ndarray:
    """silu(v) = v / (1 + e^-v) in float64 (e^-v overflows to inf for v << 0: -0)."""
    v = np.asarray(v, dtype=np.float64)
    with np.errstate(over="ignore"):
        return v / (1.0 + np.exp(-v))


def swiglu_bound(g, u, bg, bu, rel):
    """Bound on |silu(g') u' - silu(g) u| given |g' - g| <= rel*bg, |u' - u| <= rel*bu:
    |silu(g')-silu(g)| <= SILU_SLOPE*|g'-g| (mean value theorem), so the error is at most
    SILU_SLOPE*rel*bg*(|u| + rel*bu) + |silu(g)|*rel*bu."""
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    return SILU_SLOPE * rel * bg * (np.abs(u) + rel * bu) + np.abs(silu(g)) * rel * bu


def ffn_gu_matvec(qtype: int, Wg: np.ndarray, Wu: np.ndarray, N: int, K: int, x: np.ndarray,
                  rel: float = 1e-4):
    """h = silu(W_gate x) * (W_up x) for N x K gate and up weights (raw GGUF bytes).
    Returns (h, bound) float64 [B][N]; bound is swiglu_bound of the two matvec bounds."""
    g, bg = matvec(qtype, Wg, N, K, x)
    u, bu = matvec(qtype, Wu, N, K, x)
    return silu(g) * u, swiglu_bound(g, u, bg, bu, rel)


def ffn_gu_mmq(qtype: int, Wg: np.ndarray, Wu: np.ndarray, N: int, K: int, qs: np.ndarray,
               scale: np.ndarray, mrows=None, rel: float = 1e-4):
    """The MMQ form: g, u from the quantised activations (qs, scale) as in mmq()."""
    g, bg = mmq(qtype, Wg, N, K, qs, scale, mrows)
    u, bu = mmq(qtype, Wu, N, K, qs, scale, mrows)
    return silu(g) * u, swiglu_bound(g, u, bg, bu, rel)
