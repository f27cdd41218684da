"""The C-ABI library loads and exports every symbol include/r9q.h declares, and
its host-side argument checks return the documented codes without touching a
GPU (they run before any CUDA call)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._builder().build()
    return ctypes.CDLL(path)


def _declared():
    text = open(os.path.join(ROOT, "include", "r9q.h")).read()
    return sorted(set(re.findall(r"^\s*(?:int|const char\*)\s+(r9q_\w+)\s*\(", text, re.M)))


def _codes():
    text = open(os.path.join(ROOT, "include", "r9q.h")).read()
    return {k: int(v) for k, v in re.findall(r"#define\s+(R9Q_\w+)\s+(-?\d+)", text)}


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n


def test_binding_covers_header():
    import block_scaled_fp8_x128_gb300 as r9q
    for n in _declared():
        assert n in r9q.EXPORTED and callable(getattr(r9q, n)), n


def test_version_and_strerror(lib):
    c = _codes()
    lib.r9q_version.restype = ctypes.c_int
    assert lib.r9q_version() == c["R9Q_VERSION"]
    lib.r9q_strerror.restype = ctypes.c_char_p
    for k, v in c.items():
        if k.startswith("R9Q_ERR_"):
            assert lib.r9q_strerror(v) and b"unknown" not in lib.r9q_strerror(v)


def test_host_argument_checks(lib):
    c = _codes()
    P, I64, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_size_t
    f = lib.r9q_gemm_fp8_block_qa
    f.argtypes = [P, P, P, P, P, P, I64, I64, I64, P, SZ, P]
    f.restype = ctypes.c_int
    fake = 1 << 20   # never dereferenced: every case below fails before any CUDA call
    # missing weight pointer
    assert f(fake, None, None, None, fake, fake, 1, 128, 128, None, 0, None) == c["R9Q_ERR_NULL"]
    # unfused mode without aq/as
    assert f(None, None, None, fake, fake, fake, 1, 128, 128, None, 0, None) == c["R9Q_ERR_NULL"]
    # aq without as in fused mode
    assert f(fake, fake, None, fake, fake, 2 * fake, 1, 128, 128, None, 0, None) == c["R9Q_ERR_ARG"]
    # N, K not multiples of 128; M = 0
    assert f(fake, None, None, fake, fake, 4 * fake, 1, 100, 128, None, 0, None) == c["R9Q_ERR_DIM"]
    assert f(fake, None, None, fake, fake, 4 * fake, 1, 128, 200, None, 0, None) == c["R9Q_ERR_DIM"]
    assert f(fake, None, None, fake, fake, 4 * fake, 0, 128, 128, None, 0, None) == c["R9Q_ERR_DIM"]
    # misaligned activation / weight pointers
    assert f(fake + 2, None, None, 2 * fake, 3 * fake, 4 * fake, 1, 128, 128, None, 0, None) == c["R9Q_ERR_ALIGN"]
    assert f(fake, None, None, 2 * fake + 8, 3 * fake, 4 * fake, 1, 128, 128, None, 0, None) == c["R9Q_ERR_ALIGN"]
    # output aliasing the weights
    assert f(fake, None, None, 2 * fake, 3 * fake, 2 * fake, 1, 128, 128, None, 0, None) == c["R9Q_ERR_ARG"]

    g = lib.r9q_gate_up_swiglu_down
    g.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, P, P, P, ctypes.c_int, P, SZ, P]
    g.restype = ctypes.c_int
    base = [fake, 2 * fake, 3 * fake, 4 * fake, 5 * fake, 6 * fake]
    # unknown flag bits
    assert g(*base, 8, 256, 256, 256, None, None, None, 4, None, 0, None) == c["R9Q_ERR_ARG"]
    # hq without hs
    assert g(*base, 8, 256, 256, 256, None, 7 * fake, None, 0, None, 0, None) == c["R9Q_ERR_ARG"]
    # the fused path needs workspace for h when h is not an output
    assert g(*base, 8, 256, 256, 256, None, None, None, 0, None, 0, None) == c["R9Q_ERR_WORKSPACE"]
    # I not a multiple of 128
    assert g(*base, 8, 256, 200, 256, None, None, None, 0, None, 0, None) == c["R9Q_ERR_DIM"]


def test_noalloc_and_swiglu_argument_checks(lib):
    """The allocation-free MLP checks its pointers and flags before it looks at
    the device or its scratch; the SwiGLU pass checks pointers, sizes,
    alignment and overlap.  Every case fails before any CUDA call."""
    c = _codes()
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    fake = 1 << 20
    f = lib.r9q_gate_up_swiglu_down_noalloc
    f.argtypes = [P, P, P, P, P, P, I64, I64, I64, I64, P, P, ctypes.c_int, P]
    f.restype = ctypes.c_int
    base = [fake, 2 * fake, 3 * fake, 4 * fake, 5 * fake, 6 * fake]
    assert f(None, *base[1:], 8, 256, 256, 256, None, None, 0, None) == c["R9Q_ERR_NULL"]
    assert f(*base[:5], None, 8, 256, 256, 256, None, None, 0, None) == c["R9Q_ERR_NULL"]
    assert f(*base, 8, 256, 256, 256, None, None, 2, None) == c["R9Q_ERR_ARG"]          # R9Q_MLP_UNFUSED
    assert f(*base, 4096, 256, 256, 256, None, None, 0, None) == c["R9Q_ERR_WORKSPACE"]  # M*I > 524288
    g = lib.r9q_swiglu_interleaved
    g.argtypes = [P, I64, I64, P, P]
    g.restype = ctypes.c_int
    assert g(None, 2, 128, fake, None) == c["R9Q_ERR_NULL"]
    assert g(fake, 2, 100, 2 * fake, None) == c["R9Q_ERR_DIM"]
    assert g(fake, 0, 128, 2 * fake, None) == c["R9Q_ERR_DIM"]
    assert g(fake + 4, 2, 128, 2 * fake, None) == c["R9Q_ERR_ALIGN"]
    assert g(fake, 2, 128, fake + 256, None) == c["R9Q_ERR_ARG"]                  # h inside gu


def test_selftest_rejects_unknown_waits(lib):
    c = _codes()
    f = lib.r9q_selftest_wait_timeout
    f.argtypes = [ctypes.c_int, ctypes.c_void_p]
    f.restype = ctypes.c_int
    assert f(16, None) == c["R9Q_ERR_ARG"]
    assert f(-1, None) == c["R9Q_ERR_ARG"]


def test_grouped_argument_checks(lib):
    c = _codes()
    P, I64 = ctypes.c_void_p, ctypes.c_int64
    f = lib.r9q_grouped_gemm_fp8
    f.argtypes = [P, ctypes.POINTER(I64), I64, P, P, P, I64, I64, ctypes.c_int, P]
    f.restype = ctypes.c_int
    fake = 1 << 20   # never dereferenced: every case below fails (or returns) before any CUDA call

    def off(*v):
        return (I64 * len(v))(*v)
    assert f(fake, off(0, 2, 3), 2, fake, fake, 2 * fake, 128, 128, 4, None) == c["R9Q_ERR_ARG"]   # flags
    assert f(fake, None, 2, fake, fake, 2 * fake, 128, 128, 0, None) == c["R9Q_ERR_NULL"]
    assert f(fake, off(0), 0, fake, fake, 2 * fake, 128, 128, 0, None) == c["R9Q_ERR_DIM"]         # E = 0
    assert f(fake, off(*([0] * 130)), 129, fake, fake, 2 * fake, 128, 128, 0, None) == c["R9Q_ERR_DIM"]
    assert f(fake, off(1, 2, 3), 2, fake, fake, 2 * fake, 128, 128, 0, None) == c["R9Q_ERR_ARG"]   # offsets[0]
    assert f(fake, off(0, 3, 2), 2, fake, fake, 2 * fake, 128, 128, 0, None) == c["R9Q_ERR_ARG"]   # decreasing
    assert f(fake, off(0, 0, 0), 2, None, None, None, 128, 128, 0, None) == c["R9Q_OK"]           # no tokens
    assert f(fake, off(0, 1, 1), 2, None, fake, 2 * fake, 128, 128, 0, None) == c["R9Q_ERR_NULL"]
    assert f(fake, off(0, 1, 1), 2, fake, fake, 2 * fake, 100, 128, 0, None) == c["R9Q_ERR_DIM"]
    assert f(fake, off(0, 1, 1), 2, fake, fake, 2 * fake, 128, 128, 2, None) == c["R9Q_ERR_DIM"]  # SwiGLU N


def test_workspace_query(lib):
    c = _codes()
    f = lib.r9q_workspace_bytes
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_size_t)]
    f.restype = ctypes.c_int
    out = ctypes.c_size_t(123)
    assert f(c["R9Q_OP_GEMM_W8A8"], 16, 4096, 4096, 0, 0, ctypes.byref(out)) == 0 and out.value == 0
    assert f(c["R9Q_OP_GATE_UP_SWIGLU_DOWN"], 8, 1536, 4096, 4096, 0, ctypes.byref(out)) == 0
    assert out.value == 8 * 1536 * 2            # h only (already a multiple of 256)
    assert f(c["R9Q_OP_GATE_UP_SWIGLU_DOWN"], 8, 1536, 4096, 4096, c["R9Q_MLP_UNFUSED"], ctypes.byref(out)) == 0
    assert out.value == 8 * 3072 * 2 + 8 * 1536 * 2 + 8 * 1536 + 512
    assert f(99, 1, 128, 128, 0, 0, ctypes.byref(out)) == c["R9Q_ERR_ARG"]


def test_workspace_query_tensor_core_path(lib):
    """W8A8 from M = 33 on: a 64 KiB counter header, the quantised A and its
    scales, and, when few 128x256 tiles leave SMs idle, split-K partials
    (without a GPU the query plans for a GB300's 152 SMs)."""
    c = _codes()
    f = lib.r9q_workspace_bytes
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.POINTER(ctypes.c_size_t)]
    f.restype = ctypes.c_int
    out = ctypes.c_size_t(0)

    def a256(x):
        return (x + 255) // 256 * 256

    header = 64 * 1024
    # M=128 N=K=4096: 16 tiles, split-K 8 (128 CTAs): partials 16 x 8 x 128 x 256 fp32
    assert f(c["R9Q_OP_GEMM_W8A8"], 128, 4096, 4096, 0, 0, ctypes.byref(out)) == 0
    assert out.value == header + a256(128 * 4096) + a256(128 * 32 * 4) + 16 * 8 * 128 * 256 * 4
    # M=255: 32 tiles, split-K 4
    assert f(c["R9Q_OP_GEMM_W8A8"], 255, 4096, 4096, 0, 0, ctypes.byref(out)) == 0
    assert out.value == header + a256(255 * 4096) + a256(255 * 32 * 4) + 32 * 4 * 128 * 256 * 4
    # M=8192: 1024 tiles, persistent whole-K tiles, no partials
    assert f(c["R9Q_OP_GEMM_W8A8"], 8192, 4096, 4096, 0, 0, ctypes.byref(out)) == 0
    assert out.value == header + a256(8192 * 4096) + a256(8192 * 32 * 4)
    # M=32 stays on the decode stream kernel: nothing
    assert f(c["R9Q_OP_GEMM_W8A8"], 32, 4096, 4096, 0, 0, ctypes.byref(out)) == 0 and out.value == 0


def test_cpu_tensor_rejected_by_binding():
    import torch
    import block_scaled_fp8_x128_gb300 as r9q
    with pytest.raises(ValueError):
        r9q.r9q_quant_group128(torch.zeros((1, 128), dtype=torch.bfloat16))

