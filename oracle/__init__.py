"""CPU oracle for the block-scaled fp8 (e4m3) GEMM path.

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only code that may import this
package.  The product library (``block_scaled_fp8_x128_gb300``) never imports
it and shares no code with it; ``r9q_oracle.c`` is a plain C restatement of the
operation (see that file's header for the citations and the arithmetic
conventions), compiled with ``-ffp-contract=off`` so that every fp32 operation
is rounded exactly as written.

Every function here is a thin numpy <-> ctypes marshaller around the C code.
Parity pins for each function live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "r9q_oracle.c")
_LIB = os.path.join(_HERE, "libr9q_oracle.so")
_LIB_OMP = os.path.join(_HERE, "libr9q_oracle_omp.so")
_libs = {}
_all_cores = False

BLOCK = 128


def build(force: bool = False, openmp: bool = False) -> str:
    """Compile the oracle with the host C compiler (no SIMD flags, no fast
    math).  openmp=True builds the same source with -fopenmp: the GEMM loops
    then split their independent output elements over threads (used only to
    time the oracle on all host cores; the results are identical)."""
    lib = _LIB_OMP if openmp else _LIB
    if force or not os.path.exists(lib) or os.path.getmtime(lib) < os.path.getmtime(_SRC):
        tmp = lib + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               *(["-fopenmp"] if openmp else []), "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, lib)
    return lib


def use_all_cores(enable: bool = True, threads: int = 0) -> int:
    """Switch the GEMM loops to the OpenMP build (all host cores, or `threads`)
    or back to the single-threaded build; returns the thread count in use."""
    global _all_cores
    _all_cores = bool(enable)
    lib = _load()
    if enable and threads > 0:
        lib.r9o_set_threads(int(threads))
    return int(lib.r9o_threads())


def _load():
    key = _all_cores
    if key not in _libs:
        path = build(openmp=key)
        lib = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        lib.r9o_e4m3_encode.restype = ctypes.c_uint8
        lib.r9o_e4m3_encode.argtypes = [ctypes.c_float]
        lib.r9o_e4m3_decode.restype = ctypes.c_double
        lib.r9o_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.r9o_f64_to_bf16.restype = ctypes.c_uint16
        lib.r9o_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.r9o_f32_to_bf16.restype = ctypes.c_uint16
        lib.r9o_f32_to_bf16.argtypes = [ctypes.c_float]
        lib.r9o_f32_to_bf16_array.argtypes = [P, I64, P]
        lib.r9o_e4m3_encode_array.argtypes = [P, I64, P]
        lib.r9o_e4m3_encode_bits.argtypes = [ctypes.c_uint32, I64, P]
        lib.r9o_quant_group.argtypes = [P, I64, I64, I64, P, P]
        lib.r9o_quant_block128.argtypes = [P, I64, I64, P, P]
        lib.r9o_gemm_w8a8.argtypes = [P, P, P, P, I64, I64, I64, P, I64, P, P]
        lib.r9o_gemm_w8bf16.argtypes = [P, P, P, I64, I64, I64, P, I64, P, P]
        lib.r9o_swiglu_interleaved.argtypes = [P, I64, I64, P]
        lib.r9o_expf.restype = ctypes.c_float
        lib.r9o_expf.argtypes = [ctypes.c_float]
        lib.r9o_expf_array.argtypes = [P, I64, P]
        lib.r9o_silu_mul.restype = ctypes.c_float
        lib.r9o_silu_mul.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.r9o_gate_up_swiglu_down.restype = ctypes.c_int
        lib.r9o_gate_up_swiglu_down.argtypes = [P, P, P, P, P, I64, I64, I64, I64, ctypes.c_int,
                                                P, P, P, P, P]
        lib.r9o_set_threads.argtypes = [ctypes.c_int]
        lib.r9o_threads.restype = ctypes.c_int
        _libs[key] = lib
    return _libs[key]


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ scalars --

def e4m3_encode(v: float) -> int:
    """fp32 -> e4m3 code (RNE, saturating to +-448)."""
    return int(_load().r9o_e4m3_encode(float(np.float32(v))))


def e4m3_decode(code: int) -> float:
    return float(_load().r9o_e4m3_decode(int(code)))


def e4m3_decode_table() -> np.ndarray:
    """Value of every code 0..255 as float64 (NaN for 0x7F / 0xFF)."""
    return np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)


def f64_to_bf16_bits(v: float) -> int:
    return int(_load().r9o_f64_to_bf16(float(v)))


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().r9o_f32_to_bf16_array(_ptr(x), x.size, _ptr(out))
    return out


# ------------------------------------------------------------------- arrays --

def e4m3_encode_array(x: np.ndarray) -> np.ndarray:
    x = _c(x, np.float32)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().r9o_e4m3_encode_array(_ptr(x), x.size, _ptr(q))
    return q


def e4m3_encode_bits(lo: int, n: int) -> np.ndarray:
    """Codes for the fp32 bit patterns lo .. lo+n-1."""
    q = np.empty(n, dtype=np.uint8)
    _load().r9o_e4m3_encode_bits(ctypes.c_uint32(lo), n, _ptr(q))
    return q


def quant_group(x_bf16: np.ndarray, group: int = BLOCK):
    """x_bf16: uint16 bf16 bit patterns [M][K].  Returns (q uint8 [M][K], s float32 [M][K/group])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    assert K % group == 0
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, K // group), dtype=np.float32)
    _load().r9o_quant_group(_ptr(x), M, K, group, _ptr(q), _ptr(s))
    return q, s


def quant_block128(w: np.ndarray):
    """w: float32 [N][K].  Returns (q uint8 [N][K], s float32 [N/128][K/128])."""
    w = _c(w, np.float32)
    N, K = w.shape
    assert N % BLOCK == 0 and K % BLOCK == 0
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((N // BLOCK, K // BLOCK), dtype=np.float32)
    _load().r9o_quant_block128(_ptr(w), N, K, _ptr(q), _ptr(s))
    return q, s


def _rows_arg(rows, M):
    if rows is None:
        return None, M, None
    r = _c(rows, np.int64)
    assert r.ndim == 1 and (r.size == 0 or (r.min() >= 0 and r.max() < M))
    return r, r.size, _ptr(r)


def gemm_w8a8(aq, a_s, w, ws, rows=None):
    """Returns (acc float32 [R][N], y bf16 bits uint16 [R][N]); R = M or len(rows)."""
    aq, a_s, w, ws = _c(aq, np.uint8), _c(a_s, np.float32), _c(w, np.uint8), _c(ws, np.float32)
    M, K = aq.shape
    N = w.shape[0]
    assert w.shape == (N, K) and a_s.shape == (M, K // BLOCK) and ws.shape == (N // BLOCK, K // BLOCK)
    r, R, rp = _rows_arg(rows, M)
    acc = np.empty((R, N), dtype=np.float32)
    y = np.empty((R, N), dtype=np.uint16)
    _load().r9o_gemm_w8a8(_ptr(aq), _ptr(a_s), _ptr(w), _ptr(ws), M, N, K, rp, R, _ptr(acc), _ptr(y))
    return acc, y


def gemm_w8bf16(x_bf16, w, ws, rows=None):
    """Weight-only.  Returns (acc float32 [R][N], y bf16 bits uint16 [R][N])."""
    x, w, ws = _c(x_bf16, np.uint16), _c(w, np.uint8), _c(ws, np.float32)
    M, K = x.shape
    N = w.shape[0]
    assert w.shape == (N, K) and ws.shape == (N // BLOCK, K // BLOCK)
    r, R, rp = _rows_arg(rows, M)
    acc = np.empty((R, N), dtype=np.float32)
    y = np.empty((R, N), dtype=np.uint16)
    _load().r9o_gemm_w8bf16(_ptr(x), _ptr(w), _ptr(ws), M, N, K, rp, R, _ptr(acc), _ptr(y))
    return acc, y


def expf(x: np.ndarray) -> np.ndarray:
    """The oracle's fp32 exponential (Cody-Waite reduction, degree-7 Taylor
    polynomial; r9q_oracle.c) of every element of x."""
    x = _c(x, np.float32)
    y = np.empty(x.shape, dtype=np.float32)
    _load().r9o_expf_array(_ptr(x), x.size, _ptr(y))
    return y


def silu_mul(g: float, u: float) -> float:
    """silu(g) * u in fp32 as the oracle's SwiGLU step computes it (before the bf16 rounding)."""
    return float(np.float32(_load().r9o_silu_mul(float(np.float32(g)), float(np.float32(u)))))


def swiglu_interleaved(gu_bf16):
    gu = _c(gu_bf16, np.uint16)
    M, I2 = gu.shape
    h = np.empty((M, I2 // 2), dtype=np.uint16)
    _load().r9o_swiglu_interleaved(_ptr(gu), M, I2 // 2, _ptr(h))
    return h


def gate_up_swiglu_down(x_bf16, w_gu, s_gu, w_dn, s_dn, weight_only: bool = False):
    """Returns dict with gu, h (bf16 bits), hq, hs (None when weight_only), y (bf16 bits)."""
    x, w_gu, s_gu = _c(x_bf16, np.uint16), _c(w_gu, np.uint8), _c(s_gu, np.float32)
    w_dn, s_dn = _c(w_dn, np.uint8), _c(s_dn, np.float32)
    M, H = x.shape
    I = w_gu.shape[0] // 2
    Hout = w_dn.shape[0]
    assert w_gu.shape == (2 * I, H) and w_dn.shape == (Hout, I)
    gu = np.empty((M, 2 * I), dtype=np.uint16)
    h = np.empty((M, I), dtype=np.uint16)
    hq = np.empty((M, I), dtype=np.uint8)
    hs = np.empty((M, I // BLOCK), dtype=np.float32)
    y = np.empty((M, Hout), dtype=np.uint16)
    rc = _load().r9o_gate_up_swiglu_down(_ptr(x), _ptr(w_gu), _ptr(s_gu), _ptr(w_dn), _ptr(s_dn),
                                         M, H, I, Hout, int(bool(weight_only)),
                                         _ptr(gu), _ptr(h), _ptr(hq), _ptr(hs), _ptr(y))
    if rc != 0:
        raise MemoryError("oracle allocation failed")
    return {"gu": gu, "h": h, "hq": None if weight_only else hq,
            "hs": None if weight_only else hs, "y": y}


def tolerance_ok(gpu: np.ndarray, ref: np.ndarray, rel: float = 8e-3, absmax: float = 1e-3):
    """The output bound |gpu - ref| <= rel*|ref| + absmax*max|ref| per element.
    Returns (ok, worst_ratio) where worst_ratio = max |gpu-ref| / bound."""
    g = np.asarray(gpu, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    bound = rel * np.abs(r) + absmax * (np.abs(r).max() if r.size else 0.0)
    err = np.abs(g - r)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, err / bound, np.where(err > 0, np.inf, 0.0))
    worst = float(ratio.max()) if ratio.size else 0.0
    return bool(worst <= 1.0), worst
