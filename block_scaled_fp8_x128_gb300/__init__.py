"""Python binding of libr9q.so, the GB300 (sm_103a) block-scaled fp8 GEMM library.

Argument marshalling only: each function takes torch tensors, checks dtype,
shape and device, and calls the C entry point of the same name in
``include/r9q.h`` on the current CUDA stream.  Every step of the computation
runs in the library's CUDA kernels; there is no fallback.  Importing this
package raises if ``libr9q.so`` has not been built (``build.py``).
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libr9q.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libr9q.so not built at {LIB_PATH}; run block_scaled_fp8_x128_gb300/build.py")

_lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_SZ = ctypes.c_size_t

_SIGS = {
    "r9q_version": ([], ctypes.c_int),
    "r9q_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "r9q_last_device_error": ([_P], ctypes.c_int),
    "r9q_set_pdl": ([ctypes.c_int], ctypes.c_int),
    "r9q_selftest_wait_timeout": ([ctypes.c_int, _P], ctypes.c_int),
    "r9q_grouped_gemm_fp8": ([_P, ctypes.POINTER(_I64), _I64, _P, _P, _P, _I64, _I64, ctypes.c_int, _P],
                             ctypes.c_int),
    "r9q_e4m3_from_f32": ([_P, _I64, _P, _P], ctypes.c_int),
    "r9q_quant_group128": ([_P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "r9q_quant_weight_block128": ([_P, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "r9q_swiglu_interleaved": ([_P, _I64, _I64, _P, _P], ctypes.c_int),
    "r9q_gemm_fp8_block_qa": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "r9q_gemm_fp8w_bf16a": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "r9q_gate_up_swiglu_down": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, _P, ctypes.c_int,
                                 _P, _SZ, _P], ctypes.c_int),
    "r9q_workspace_bytes": ([ctypes.c_int, _I64, _I64, _I64, _I64, ctypes.c_int, ctypes.POINTER(_SZ)],
                            ctypes.c_int),
    "r9q_gate_up_swiglu_down_noalloc": ([_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _P, _P, ctypes.c_int, _P],
                                        ctypes.c_int),
}
for _name, (_args, _res) in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = _res

EXPORTED = tuple(_SIGS)

R9Q_ERR_TIMEOUT = -6
R9Q_GROUPED_WEIGHT_ONLY = 1
R9Q_GROUPED_SWIGLU = 2
R9Q_MLP_WEIGHT_ONLY = 1
R9Q_MLP_UNFUSED = 2
R9Q_OP_GEMM_W8A8 = 1
R9Q_OP_GEMM_W8BF16 = 2
R9Q_OP_GATE_UP_SWIGLU_DOWN = 3


class R9QError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({_lib.r9q_strerror(code).decode()})")


def _check(rc: int, where: str) -> None:
    if rc != 0:
        raise R9QError(rc, where)


def _ptr(t: torch.Tensor | None):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("tensor must be on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _expect(t, dtype, shape, name):
    if t is None:
        return
    if t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: expected shape {tuple(shape)}, got {tuple(t.shape)}")


def r9q_version() -> int:
    return int(_lib.r9q_version())


def r9q_strerror(code: int) -> str:
    return _lib.r9q_strerror(int(code)).decode()


def r9q_grouped_gemm_fp8(a: torch.Tensor, offsets, w: torch.Tensor, ws: torch.Tensor, y: torch.Tensor | None = None,
                         flags: int = 0, stream=None) -> torch.Tensor:
    """Several experts in one launch: a bf16 [offsets[-1]][K] (tokens sorted by
    expert), offsets host ints [E + 1], w e4m3 [E][N][K], ws fp32
    [E][N/128][K/128]; y bf16 [offsets[-1]][N] (N/2 with R9Q_GROUPED_SWIGLU)."""
    off = [int(v) for v in offsets]
    E = len(off) - 1
    Mtot, K = a.shape
    _expect(a, torch.bfloat16, (off[-1], K), "a")
    if w.dim() != 3 or w.shape[0] != E or w.shape[2] != K:
        raise ValueError("w must be [E][N][K]")
    N = w.shape[1]
    _expect(w, torch.uint8, (E, N, K), "w")
    _expect(ws, torch.float32, (E, N // 128, K // 128), "ws")
    ncols = N // 2 if flags & R9Q_GROUPED_SWIGLU else N
    if y is None:
        y = torch.empty((Mtot, ncols), dtype=torch.bfloat16, device=a.device)
    _expect(y, torch.bfloat16, (Mtot, ncols), "y")
    arr = (_I64 * (E + 1))(*off)
    _check(_lib.r9q_grouped_gemm_fp8(_ptr(a), arr, E, _ptr(w), _ptr(ws), _ptr(y), N, K, int(flags), _stream(stream)),
           "r9q_grouped_gemm_fp8")
    return y


def r9q_selftest_wait_timeout(which: int, stream=None) -> None:
    """Launch the failure-detection self-test kernel (its bounded waits run
    out and record R9Q_ERR_TIMEOUT; read it with r9q_last_device_error)."""
    _check(_lib.r9q_selftest_wait_timeout(int(which), _stream(stream)), "r9q_selftest_wait_timeout")


def r9q_set_pdl(enable: bool) -> bool:
    """Programmatic dependent launch for the GEMMs (see include/r9q.h); returns the previous setting."""
    return bool(_lib.r9q_set_pdl(int(bool(enable))))


def r9q_last_device_error(stream=None) -> int:
    rc = int(_lib.r9q_last_device_error(_stream(stream)))
    if rc != 0:
        # a kernel gave up mid-call: its workspace counters may be left non-zero
        _WORKSPACES.clear()
    return rc


# One zero-filled W8A8 workspace per (device, stream) for calls that pass
# none.  Every call that completes leaves the workspace's counter header at
# zero again, so the same tensor serves every later call on that stream
# (calls on one stream are ordered); it grows when a larger call needs more.
_WORKSPACES: dict = {}


def _stream_workspace(need: int, device: torch.device, stream=None) -> torch.Tensor:
    s = stream if stream is not None else torch.cuda.current_stream(device)
    key = (device.index, s.cuda_stream)
    ws = _WORKSPACES.get(key)
    if ws is None or ws.numel() < need:
        ws = torch.zeros(need, dtype=torch.uint8, device=device)
        _WORKSPACES[key] = ws
    return ws


def r9q_e4m3_from_f32(x: torch.Tensor, q: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    _expect(x, torch.float32, x.shape, "x")
    if q is None:
        q = torch.empty(x.shape, dtype=torch.uint8, device=x.device)
    _expect(q, torch.uint8, x.shape, "q")
    _check(_lib.r9q_e4m3_from_f32(_ptr(x), x.numel(), _ptr(q), _stream(stream)), "r9q_e4m3_from_f32")
    return q


def r9q_quant_group128(x: torch.Tensor, xq: torch.Tensor | None = None, xs: torch.Tensor | None = None,
                       stream=None):
    M, K = x.shape
    _expect(x, torch.bfloat16, (M, K), "x")
    if xq is None:
        xq = torch.empty((M, K), dtype=torch.uint8, device=x.device)
    if xs is None:
        xs = torch.empty((M, K // 128), dtype=torch.float32, device=x.device)
    _expect(xq, torch.uint8, (M, K), "xq")
    _expect(xs, torch.float32, (M, K // 128), "xs")
    _check(_lib.r9q_quant_group128(_ptr(x), M, K, _ptr(xq), _ptr(xs), _stream(stream)), "r9q_quant_group128")
    return xq, xs


def r9q_swiglu_interleaved(gu: torch.Tensor, h: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """gu bf16 [M][2I] (gate/up interleaved per 128 columns) -> h bf16 [M][I]."""
    M, I2 = gu.shape
    I = I2 // 2
    _expect(gu, torch.bfloat16, (M, 2 * I), "gu")
    if h is None:
        h = torch.empty((M, I), dtype=torch.bfloat16, device=gu.device)
    _expect(h, torch.bfloat16, (M, I), "h")
    _check(_lib.r9q_swiglu_interleaved(_ptr(gu), M, I, _ptr(h), _stream(stream)), "r9q_swiglu_interleaved")
    return h


def r9q_quant_weight_block128(w: torch.Tensor, wq: torch.Tensor | None = None, ws: torch.Tensor | None = None,
                              stream=None):
    N, K = w.shape
    _expect(w, torch.float32, (N, K), "w")
    if wq is None:
        wq = torch.empty((N, K), dtype=torch.uint8, device=w.device)
    if ws is None:
        ws = torch.empty((N // 128, K // 128), dtype=torch.float32, device=w.device)
    _expect(wq, torch.uint8, (N, K), "wq")
    _expect(ws, torch.float32, (N // 128, K // 128), "ws")
    _check(_lib.r9q_quant_weight_block128(_ptr(w), N, K, _ptr(wq), _ptr(ws), _stream(stream)),
           "r9q_quant_weight_block128")
    return wq, ws


def r9q_workspace_bytes(op: int, M: int, N: int, K: int, N2: int = 0, flags: int = 0) -> int:
    out = _SZ(0)
    _check(_lib.r9q_workspace_bytes(int(op), M, N, K, N2, int(flags), ctypes.byref(out)), "r9q_workspace_bytes")
    return int(out.value)


def r9q_gemm_fp8_block_qa(a: torch.Tensor | None, w: torch.Tensor, ws: torch.Tensor,
                          y: torch.Tensor | None = None, aq: torch.Tensor | None = None,
                          as_: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                          M: int | None = None, stream=None) -> torch.Tensor:
    """W8A8.  a (bf16 [M][K]) given: fused quant, aq/as_ optional outputs.
    a None: aq (uint8 [M][K]) / as_ (fp32 [M][K/128]) are the inputs.
    workspace: uint8 device tensor of at least r9q_workspace_bytes(R9Q_OP_GEMM_W8A8, M, N, K)
    bytes, zero-filled before its first use (e.g. torch.zeros); the calls keep its counter
    header at zero, so one workspace serves any sequence of calls on one stream.  When omitted,
    the binding reuses one zeroed workspace per (device, stream), allocated (and zero-filled)
    on the first call that needs it or needs more; pass your own to control that allocation,
    e.g. before capturing a CUDA graph."""
    N, K = w.shape
    src = a if a is not None else aq
    if src is None:
        raise ValueError("need a or aq/as_")
    M = src.shape[0]
    _expect(a, torch.bfloat16, (M, K), "a")
    _expect(aq, torch.uint8, (M, K), "aq")
    _expect(as_, torch.float32, (M, K // 128), "as")
    _expect(w, torch.uint8, (N, K), "w")
    _expect(ws, torch.float32, (N // 128, K // 128), "ws")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=w.device)
    _expect(y, torch.bfloat16, (M, N), "y")
    if workspace is None:
        need = r9q_workspace_bytes(R9Q_OP_GEMM_W8A8, M, N, K)
        if need:
            workspace = _stream_workspace(need, w.device, stream)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.r9q_gemm_fp8_block_qa(_ptr(a), _ptr(aq), _ptr(as_), _ptr(w), _ptr(ws), _ptr(y), M, N, K,
                                      _ptr(workspace), wsb, _stream(stream)), "r9q_gemm_fp8_block_qa")
    return y


def r9q_gemm_fp8w_bf16a(a: torch.Tensor, w: torch.Tensor, ws: torch.Tensor, y: torch.Tensor | None = None,
                        workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M, K = a.shape
    N = w.shape[0]
    _expect(a, torch.bfloat16, (M, K), "a")
    _expect(w, torch.uint8, (N, K), "w")
    _expect(ws, torch.float32, (N // 128, K // 128), "ws")
    if y is None:
        y = torch.empty((M, N), dtype=torch.bfloat16, device=w.device)
    _expect(y, torch.bfloat16, (M, N), "y")
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.r9q_gemm_fp8w_bf16a(_ptr(a), _ptr(w), _ptr(ws), _ptr(y), M, N, K, _ptr(workspace), wsb,
                                    _stream(stream)), "r9q_gemm_fp8w_bf16a")
    return y


def r9q_gate_up_swiglu_down(x: torch.Tensor, w_gu: torch.Tensor, s_gu: torch.Tensor, w_dn: torch.Tensor,
                            s_dn: torch.Tensor, y: torch.Tensor | None = None, h: torch.Tensor | None = None,
                            hq: torch.Tensor | None = None, hs: torch.Tensor | None = None, flags: int = 0,
                            workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    M, H = x.shape
    I = w_gu.shape[0] // 2
    H_out = w_dn.shape[0]
    _expect(x, torch.bfloat16, (M, H), "x")
    _expect(w_gu, torch.uint8, (2 * I, H), "w_gu")
    _expect(s_gu, torch.float32, (2 * I // 128, H // 128), "s_gu")
    _expect(w_dn, torch.uint8, (H_out, I), "w_dn")
    _expect(s_dn, torch.float32, (H_out // 128, I // 128), "s_dn")
    _expect(h, torch.bfloat16, (M, I), "h")
    _expect(hq, torch.uint8, (M, I), "hq")
    _expect(hs, torch.float32, (M, I // 128), "hs")
    if y is None:
        y = torch.empty((M, H_out), dtype=torch.bfloat16, device=x.device)
    _expect(y, torch.bfloat16, (M, H_out), "y")
    if workspace is None:
        need = r9q_workspace_bytes(R9Q_OP_GATE_UP_SWIGLU_DOWN, M, I, H, H_out, flags)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=x.device)
    wsb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib.r9q_gate_up_swiglu_down(_ptr(x), _ptr(w_gu), _ptr(s_gu), _ptr(w_dn), _ptr(s_dn), _ptr(y),
                                        M, H, I, H_out, _ptr(h), _ptr(hq), _ptr(hs), int(flags),
                                        _ptr(workspace), wsb, _stream(stream)), "r9q_gate_up_swiglu_down")
    return y


def r9q_gate_up_swiglu_down_noalloc(x: torch.Tensor, w_gu: torch.Tensor, s_gu: torch.Tensor, w_dn: torch.Tensor,
                                    s_dn: torch.Tensor, y: torch.Tensor | None = None,
                                    hq: torch.Tensor | None = None, hs: torch.Tensor | None = None,
                                    flags: int = 0, stream=None) -> torch.Tensor:
    """The fused expert MLP without workspace (h lives in the library's fixed
    scratch; see include/r9q.h for the size limit and the sharing rules)."""
    M, H = x.shape
    I = w_gu.shape[0] // 2
    H_out = w_dn.shape[0]
    _expect(x, torch.bfloat16, (M, H), "x")
    _expect(w_gu, torch.uint8, (2 * I, H), "w_gu")
    _expect(s_gu, torch.float32, (2 * I // 128, H // 128), "s_gu")
    _expect(w_dn, torch.uint8, (H_out, I), "w_dn")
    _expect(s_dn, torch.float32, (H_out // 128, I // 128), "s_dn")
    _expect(hq, torch.uint8, (M, I), "hq")
    _expect(hs, torch.float32, (M, I // 128), "hs")
    if y is None:
        y = torch.empty((M, H_out), dtype=torch.bfloat16, device=x.device)
    _expect(y, torch.bfloat16, (M, H_out), "y")
    _check(_lib.r9q_gate_up_swiglu_down_noalloc(_ptr(x), _ptr(w_gu), _ptr(s_gu), _ptr(w_dn), _ptr(s_dn), _ptr(y),
                                                M, H, I, H_out, _ptr(hq), _ptr(hs), int(flags), _stream(stream)),
           "r9q_gate_up_swiglu_down_noalloc")
    return y
