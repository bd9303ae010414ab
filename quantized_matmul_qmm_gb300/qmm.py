"""Thin ctypes binding of libqmm (include/qmm.h).

Argument marshalling only.  Every step of the computation runs in the CUDA
library.  The functions take torch tensors for device memory and use torch's
current CUDA stream.  Each one raises ``QmmError`` when the C entry point
returns a status other than QMM_OK.  There is no Python fallback: if
libqmm.so is missing, importing this module raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libqmm.so")

QMM_OK, QMM_ERR_INVALID_ARG, QMM_ERR_UNSUPPORTED, QMM_ERR_OVERFLOW_BOUND = 0, 1, 2, 3
QMM_ERR_CUDA, QMM_ERR_TIMEOUT, QMM_ERR_BAD_EXPERT_ID, QMM_ERR_WORKSPACE, QMM_ERR_RANGE = 4, 5, 6, 7, 8
QMM_U8, QMM_S8, QMM_S32, QMM_F32, QMM_BF16 = 1, 2, 3, 4, 5
DTYPES = {"u8": QMM_U8, "s8": QMM_S8, "s32": QMM_S32, "f32": QMM_F32, "bf16": QMM_BF16}
TORCH_OUT = {"s32": torch.int32, "f32": torch.float32, "s8": torch.int8, "u8": torch.uint8}

# exported symbols and their C signatures (restype, argtypes)
_c = ctypes
_vp, _i64, _i32, _sz = _c.c_void_p, _c.c_int64, _c.c_int32, _c.c_size_t
_szp = _c.POINTER(_c.c_size_t)


class QmmEpilogue(ctypes.Structure):
    _fields_ = [("out_type", _c.c_int), ("bias", _vp), ("s_x", _vp), ("s_x_stride", _i64),
                ("s_w", _vp), ("s_y", _c.c_float), ("zp_y", _i32)]


class QmmInt8Problem(ctypes.Structure):
    _fields_ = [("A", _vp), ("a_type", _c.c_int), ("M", _i64), ("K", _i64), ("lda", _i64), ("zA", _i32),
                ("packedB", _vp), ("col_sum", _vp), ("N", _i64), ("b_orig_type", _c.c_int), ("zB", _i32),
                ("ep", QmmEpilogue), ("out", _vp), ("ldo", _i64)]


class QmmQ4GemvProblem(ctypes.Structure):
    _fields_ = [("tiles", _vp), ("N", _i64), ("K", _i64), ("x", _vp), ("y", _vp)]


SIGNATURES = {
    "qmm_status_string": (_c.c_char_p, [_c.c_int]),
    "qmm_version": (_c.c_int, []),
    "qmm_pack_b_int8_size": (_c.c_int, [_i64, _i64, _szp]),
    "qmm_pack_b_int8": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _i64, _vp, _sz, _vp, _vp, _vp]),
    "qmm_int8_gemm_workspace_size": (_c.c_int, [_i64, _i64, _i64, _szp]),
    "qmm_int8_gemm": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _i64, _i32, _vp, _vp, _i64, _c.c_int,
                                 _i32, _c.POINTER(QmmEpilogue), _vp, _i64, _vp, _sz, _vp, _vp]),
    "qmm_widen_b_int8_size": (_c.c_int, [_i64, _i64, _szp]),
    "qmm_widen_b_int8": (_c.c_int, [_vp, _i64, _i64, _vp, _sz, _vp, _vp]),
    "qmm_int8_gemm_b16_workspace_size": (_c.c_int, [_i64, _i64, _i64, _szp]),
    "qmm_int8_gemm_b16": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _i64, _i32, _vp, _vp, _vp, _i64, _c.c_int,
                                     _i32, _c.POINTER(QmmEpilogue), _vp, _i64, _vp, _sz, _vp, _vp]),
    "qmm_int8_gemm_group": (_c.c_int, [_c.POINTER(QmmInt8Problem), _i64, _vp, _vp]),
    "qmm_int8_gemm_axis_zp_workspace_size": (_c.c_int, [_i64, _i64, _i64, _szp]),
    "qmm_int8_gemm_axis_zp": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _i64, _vp, _vp, _vp, _i64, _c.c_int,
                                         _vp, _c.POINTER(QmmEpilogue), _vp, _i64, _vp, _sz, _vp, _vp]),
    "qmm_quantize_act_int8_workspace_size": (_c.c_int, [_i64, _i64, _c.c_int, _szp]),
    "qmm_quantize_act_int8": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _i64, _c.c_int, _vp, _i64, _vp, _vp, _sz,
                                         _vp]),
    "qmm_pack_q4_size": (_c.c_int, [_i64, _i64, _szp]),
    "qmm_pack_q4": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "qmm_q4_gemm_workspace_size": (_c.c_int, [_i64, _i64, _i64, _szp]),
    "qmm_q4_gemm": (_c.c_int, [_vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _sz, _vp, _vp]),
    "qmm_q4_gemv_group": (_c.c_int, [_c.POINTER(QmmQ4GemvProblem), _i64, _vp, _vp]),
    "qmm_q4_gemm_id_workspace_size": (_c.c_int, [_i64, _i64, _i64, _i64, _szp]),
    "qmm_q4_gemm_id": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64, _i64,
                                  _vp, _i64, _i64, _vp, _sz, _vp, _vp]),
    "qmm_q4_gemm_id_pair": (_c.c_int, [_vp, _vp, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _i64, _i64, _vp, _vp,
                                       _i64, _i64, _vp, _sz, _vp, _vp]),
    "qmm_q4_gemm_id_noalloc": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _i64,
                                          _i64, _vp, _i64, _i64, _vp, _vp]),
    "qmm_pack_w8_size": (_c.c_int, [_i64, _i64, _szp, _szp]),
    "qmm_pack_w8": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _sz, _vp, _sz, _vp]),
    "qmm_w8_gemm_workspace_size": (_c.c_int, [_i64, _i64, _i64, _szp]),
    "qmm_w8_gemm": (_c.c_int, [_vp, _vp, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _sz, _vp, _vp]),
    "qmm_repack_q4k": (_c.c_int, [_vp, _i64, _i64, _i64, _vp, _sz, _vp]),
    "qmm_pack_q8_size": (_c.c_int, [_i64, _i64, _szp]),
    "qmm_pack_q8": (_c.c_int, [_vp, _i64, _i64, _i64, _c.c_int, _vp, _sz, _vp]),
    "qmm_q8_gemm_workspace_size": (_c.c_int, [_i64, _i64, _i64, _szp]),
    "qmm_q8_gemm": (_c.c_int, [_vp, _c.c_int, _i64, _i64, _vp, _i64, _i64, _vp, _i64, _vp, _sz, _vp, _vp]),
    "qmm_probe_hbm_read": (_c.c_int, [_vp, _sz, _c.c_int, _vp, _vp, _vp]),
    "qmm_selftest_wait_timeout": (_c.c_int, [_c.c_uint64, _vp, _vp, _vp]),
}
QMM_Q8_LAYOUT_KR, QMM_Q8_LAYOUT_SLAB16 = 0, 1


class QmmError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        super().__init__(f"{fn} returned {status_string(status)} ({status})")


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libqmm.so not built ({path}); run quantized_matmul_qmm_gb300.build.build()")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    return lib


lib = load_library()


def status_string(s: int) -> str:
    return lib.qmm_status_string(int(s)).decode()


def _check(fn: str, status: int):
    if status != QMM_OK:
        raise QmmError(fn, status)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _size(fn, *args) -> int:
    out = ctypes.c_size_t(0)
    _check(fn, getattr(lib, fn)(*args, ctypes.byref(out)))
    return int(out.value)


# ---------------------------------------------------------------------------
# int8
# ---------------------------------------------------------------------------

def pack_b_int8_size(K: int, N: int) -> int:
    return _size("qmm_pack_b_int8_size", K, N)


def pack_b_int8(B: torch.Tensor, b_type: str):
    """B: device [K][N] (fp32, int8 or uint8).  Returns (packed [N][Kp] int8,
    col_scale [N] fp32 or None, col_sum [N] int32)."""
    K, N = B.shape
    dev = B.device
    nbytes = pack_b_int8_size(K, N)
    packed = torch.empty(nbytes, dtype=torch.int8, device=dev).view(N, nbytes // N)
    col_scale = torch.empty(N, dtype=torch.float32, device=dev) if b_type == "f32" else None
    col_sum = torch.empty(N, dtype=torch.int32, device=dev)
    _check("qmm_pack_b_int8", lib.qmm_pack_b_int8(
        _ptr(B), DTYPES[b_type], K, N, B.stride(0), _ptr(packed), nbytes, _ptr(col_scale),
        _ptr(col_sum), _stream()))
    return packed, col_scale, col_sum


def int8_gemm_workspace_size(M: int, K: int, N: int) -> int:
    return _size("qmm_int8_gemm_workspace_size", M, K, N)


def widen_b_int8(packed: torch.Tensor, K: int, N: int, dev_status=None) -> torch.Tensor:
    """packed [N][Kp] int8 from pack_b_int8 -> its f16 copy [N][Kp] through
    qmm_widen_b_int8 (done once, like the pack)."""
    nbytes = _size("qmm_widen_b_int8_size", K, N)
    b16 = torch.empty(nbytes // 2, dtype=torch.float16, device=packed.device).view(N, nbytes // (2 * N))
    _check("qmm_widen_b_int8", lib.qmm_widen_b_int8(_ptr(packed), K, N, _ptr(b16), nbytes, _ptr(dev_status),
                                                    _stream()))
    return b16


def int8_gemm(A: torch.Tensor, a_type: str, zA: int, packed: torch.Tensor, col_sum: torch.Tensor,
              N: int, b_orig_type: str, zB: int, out_type: str = "s32", bias=None, s_x=None,
              s_x_stride: int = 0, s_w=None, s_y: float = 1.0, zp_y: int = 0, out=None,
              workspace=None, dev_status=None, b16=None):
    """Y = A (x) packB through qmm_int8_gemm, or qmm_int8_gemm_b16 when b16
    (from widen_b_int8) is given.  Returns the output tensor."""
    M, K = A.shape
    if out is None:
        out = torch.empty((M, N), dtype=TORCH_OUT[out_type], device=A.device)
    ws_need = (_size("qmm_int8_gemm_b16_workspace_size", M, K, N) if b16 is not None
               else int8_gemm_workspace_size(M, K, N))
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=A.device)
    ep = QmmEpilogue(DTYPES[out_type], _ptr(bias), _ptr(s_x), s_x_stride, _ptr(s_w),
                     float(s_y), int(zp_y))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    if b16 is not None:
        _check("qmm_int8_gemm_b16", lib.qmm_int8_gemm_b16(
            _ptr(A), DTYPES[a_type], M, K, A.stride(0), int(zA), _ptr(packed), _ptr(b16), _ptr(col_sum), N,
            DTYPES[b_orig_type], int(zB), ctypes.byref(ep), _ptr(out), out.stride(0), _ptr(workspace), ws_bytes,
            _ptr(dev_status), _stream()))
        return out
    _check("qmm_int8_gemm", lib.qmm_int8_gemm(
        _ptr(A), DTYPES[a_type], M, K, A.stride(0), int(zA), _ptr(packed), _ptr(col_sum), N,
        DTYPES[b_orig_type], int(zB), ctypes.byref(ep), _ptr(out), out.stride(0), _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream()))
    return out


def int8_gemm_group(problems, dev_status=None):
    """Several small-M int8 GEMMs (M <= 64) in one launch through
    qmm_int8_gemm_group.  problems: list of dicts with int8_gemm's arguments
    (A, a_type, zA, packed, col_sum, N, b_orig_type, zB, out_type, bias, s_x,
    s_x_stride, s_w, s_y, zp_y, out); `out` is created when absent.  Returns
    the list of outputs."""
    arr = (QmmInt8Problem * len(problems))()
    outs = []
    for i, d in enumerate(problems):
        A = d["A"]
        M, K = A.shape
        N, ot = d["N"], d.get("out_type", "s32")
        out = d.get("out")
        if out is None:
            out = torch.empty((M, N), dtype=TORCH_OUT[ot], device=A.device)
        outs.append(out)
        ep = QmmEpilogue(DTYPES[ot], _ptr(d.get("bias")), _ptr(d.get("s_x")), d.get("s_x_stride", 0),
                         _ptr(d.get("s_w")), float(d.get("s_y", 1.0)), int(d.get("zp_y", 0)))
        ptr = lambda t: 0 if t is None else t.data_ptr()
        arr[i] = QmmInt8Problem(ptr(A), DTYPES[d["a_type"]], M, K, A.stride(0), int(d["zA"]), ptr(d["packed"]),
                                ptr(d["col_sum"]), N, DTYPES[d["b_orig_type"]], int(d["zB"]), ep, ptr(out),
                                out.stride(0))
    _check("qmm_int8_gemm_group", lib.qmm_int8_gemm_group(arr, len(problems), _ptr(dev_status), _stream()))
    return outs


def int8_gemm_axis_zp_workspace_size(M: int, K: int, N: int) -> int:
    return _size("qmm_int8_gemm_axis_zp_workspace_size", M, K, N)


def int8_gemm_axis_zp(A: torch.Tensor, a_type: str, zA, packed: torch.Tensor, col_sum: torch.Tensor,
                      N: int, b_orig_type: str, zB, out_type: str = "s32", bias=None, s_x=None,
                      s_x_stride: int = 0, s_w=None, s_y: float = 1.0, zp_y: int = 0, out=None,
                      workspace=None, dev_status=None):
    """qmm_int8_gemm with per-axis zero points: zA a device int32 [M] (or None:
    all 0), zB a device int32 [N] (or None).  Returns the output tensor."""
    M, K = A.shape
    if out is None:
        out = torch.empty((M, N), dtype=TORCH_OUT[out_type], device=A.device)
    if workspace is None:
        workspace = torch.empty(int8_gemm_axis_zp_workspace_size(M, K, N), dtype=torch.uint8, device=A.device)
    ep = QmmEpilogue(DTYPES[out_type], _ptr(bias), _ptr(s_x), s_x_stride, _ptr(s_w),
                     float(s_y), int(zp_y))
    _check("qmm_int8_gemm_axis_zp", lib.qmm_int8_gemm_axis_zp(
        _ptr(A), DTYPES[a_type], M, K, A.stride(0), _ptr(zA), _ptr(packed), _ptr(col_sum), N,
        DTYPES[b_orig_type], _ptr(zB), ctypes.byref(ep), _ptr(out), out.stride(0), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream()))
    return out


def quantize_act_int8_workspace_size(M: int, K: int, per_row: bool) -> int:
    return _size("qmm_quantize_act_int8_workspace_size", M, K, int(per_row))


def quantize_act_int8(X: torch.Tensor, per_row: bool = True, A=None, s_x=None, workspace=None):
    """Symmetric int8 codes of X (fp32 or bf16 [M][K] on the device) through
    qmm_quantize_act_int8.  Returns (A int8 [M][K], s_x fp32 [M] or [1])."""
    M, K = X.shape
    x_type = {torch.float32: "f32", torch.bfloat16: "bf16"}[X.dtype]
    if A is None:
        lda = (K + 15) // 16 * 16
        A = torch.empty((M, lda), dtype=torch.int8, device=X.device)[:, :K]
    if s_x is None:
        s_x = torch.empty(M if per_row else 1, dtype=torch.float32, device=X.device)
    ws_need = quantize_act_int8_workspace_size(M, K, per_row)
    if workspace is None and ws_need > 0:
        workspace = torch.empty(ws_need, dtype=torch.uint8, device=X.device)
    _check("qmm_quantize_act_int8", lib.qmm_quantize_act_int8(
        _ptr(X), DTYPES[x_type], M, K, X.stride(0), int(per_row), _ptr(A), A.stride(0), _ptr(s_x),
        _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(), _stream()))
    return A, s_x


# ---------------------------------------------------------------------------
# 4-bit
# ---------------------------------------------------------------------------

def pack_q4_size(N: int, K: int) -> int:
    return _size("qmm_pack_q4_size", N, K)


def pack_q4(W: torch.Tensor) -> torch.Tensor:
    """W: device fp32 [N][K].  Returns the tile bytes (uint8)."""
    N, K = W.shape
    nbytes = pack_q4_size(N, K)
    tiles = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _check("qmm_pack_q4", lib.qmm_pack_q4(_ptr(W), N, K, W.stride(0), _ptr(tiles), nbytes,
                                          _stream()))
    return tiles


def q4_gemm_workspace_size(M: int, K: int, N: int) -> int:
    return _size("qmm_q4_gemm_workspace_size", M, K, N)


def q4_gemm(tiles: torch.Tensor, N: int, K: int, X: torch.Tensor, Y=None, workspace=None, dev_status=None):
    """Y[m][n] = sum_k X[m][k] w[n][k]; X bf16 [M][K] on the device."""
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    if workspace is None:
        need = q4_gemm_workspace_size(M, K, N)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    _check("qmm_q4_gemm", lib.qmm_q4_gemm(
        _ptr(tiles), N, K, _ptr(X), M, X.stride(0), _ptr(Y), Y.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream()))
    return Y


def q4_gemv_group(problems, dev_status=None):
    """Grouped decode GEMVs in one launch: problems is a list of
    (tiles, N, K, x, y) with x bf16 [K] and y fp32 [N] on the device;
    y_i = W_i x_i for every i.  Returns the list of y tensors."""
    arr = (QmmQ4GemvProblem * len(problems))()
    for i, (tiles, N, K, x, y) in enumerate(problems):
        arr[i] = QmmQ4GemvProblem(tiles.data_ptr(), N, K, x.data_ptr(), y.data_ptr())
    _check("qmm_q4_gemv_group", lib.qmm_q4_gemv_group(arr, len(problems), _ptr(dev_status), _stream()))
    return [y for (_, _, _, _, y) in problems]


def q4_gemm_id_workspace_size(n_expert: int, n_used: int, T: int, K: int) -> int:
    return _size("qmm_q4_gemm_id_workspace_size", n_expert, n_used, T, K)


def q4_gemm_id(tiles: torch.Tensor, n_expert: int, N: int, K: int, X: torch.Tensor,
               ids: torch.Tensor, ld_ids: int, n_used: int, T: int, Y=None, workspace=None,
               dev_status=None):
    """MUL_MAT_ID.  X is [T][K] (shared src1) or [T][n_used][K] (per-slot src1);
    ids a device int32 buffer read as ids[t*ld_ids + i].  Returns Y [T][n_used][N]."""
    if X.dim() == 2:
        ldx_token, ldx_slot = X.stride(0), 0
    else:
        ldx_token, ldx_slot = X.stride(0), X.stride(1)
    if Y is None:
        Y = torch.empty((T, n_used, N), dtype=torch.float32, device=X.device)
    if workspace is None:
        workspace = torch.empty(q4_gemm_id_workspace_size(n_expert, n_used, T, K), dtype=torch.uint8,
                                device=X.device)
    _check("qmm_q4_gemm_id", lib.qmm_q4_gemm_id(
        _ptr(tiles), n_expert, N, K, _ptr(X), ldx_token, ldx_slot, _ptr(ids), ld_ids, n_used, T,
        _ptr(Y), Y.stride(0), Y.stride(1), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream()))
    return Y


def q4_gemm_id_pair(tiles_gate: torch.Tensor, tiles_up: torch.Tensor, n_expert: int, N: int, K: int,
                    X: torch.Tensor, ids: torch.Tensor, ld_ids: int, n_used: int, T: int, Y_gate=None, Y_up=None,
                    workspace=None, dev_status=None):
    """The gate/up pair: both MUL_MAT_IDs over the shared src1 X [T][K] in one
    call.  Returns (Y_gate, Y_up), each [T][n_used][N]."""
    if Y_gate is None:
        Y_gate = torch.empty((T, n_used, N), dtype=torch.float32, device=X.device)
    if Y_up is None:
        Y_up = torch.empty((T, n_used, N), dtype=torch.float32, device=X.device)
    assert Y_gate.stride() == Y_up.stride()
    if workspace is None:
        workspace = torch.empty(q4_gemm_id_workspace_size(n_expert, n_used, T, K), dtype=torch.uint8,
                                device=X.device)
    _check("qmm_q4_gemm_id_pair", lib.qmm_q4_gemm_id_pair(
        _ptr(tiles_gate), _ptr(tiles_up), n_expert, N, K, _ptr(X), X.stride(0), _ptr(ids), ld_ids, n_used, T,
        _ptr(Y_gate), _ptr(Y_up), Y_gate.stride(0), Y_gate.stride(1), _ptr(workspace),
        workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream()))
    return Y_gate, Y_up


def q4_gemm_id_noalloc(tiles: torch.Tensor, n_expert: int, N: int, K: int, X: torch.Tensor,
                       ids: torch.Tensor, ld_ids: int, n_used: int, T: int, Y: torch.Tensor,
                       dev_status=None):
    """MUL_MAT_ID through qmm_q4_gemm_id_noalloc: the same result as
    q4_gemm_id, for callers that cannot allocate device memory.  The library
    keeps the routing tables and activation-row scales in its own fixed device
    array (and packs the activation rows there when they fit), so the caller
    passes only inputs and the output Y [T][n_used][N] (preallocated).
    Limits: n_expert <= 1024, T * n_used <= 65536."""
    if X.dim() == 2:
        ldx_token, ldx_slot = X.stride(0), 0
    else:
        ldx_token, ldx_slot = X.stride(0), X.stride(1)
    _check("qmm_q4_gemm_id_noalloc", lib.qmm_q4_gemm_id_noalloc(
        _ptr(tiles), n_expert, N, K, _ptr(X), ldx_token, ldx_slot, _ptr(ids), ld_ids, n_used, T,
        _ptr(Y), Y.stride(0), Y.stride(1), _ptr(dev_status), _stream()))
    return Y


# ---------------------------------------------------------------------------
# W8A16
# ---------------------------------------------------------------------------

def pack_w8_size(N: int, K: int):
    """(code bytes, scale bytes) of an N x K weight."""
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    _check("qmm_pack_w8_size", lib.qmm_pack_w8_size(N, K, ctypes.byref(cb), ctypes.byref(sb)))
    return int(cb.value), int(sb.value)


def pack_w8(W: torch.Tensor):
    """W: device fp32 [N][K].  Returns (codes int8 [N][Kp], scales fp32 [N][ceil(K/1024)])."""
    N, K = W.shape
    cb, sb = pack_w8_size(N, K)
    codes = torch.empty((N, cb // N), dtype=torch.int8, device=W.device)
    scales = torch.empty((N, sb // (4 * N)), dtype=torch.float32, device=W.device)
    _check("qmm_pack_w8", lib.qmm_pack_w8(_ptr(W), N, K, W.stride(0), _ptr(codes), cb, _ptr(scales), sb,
                                          _stream()))
    return codes, scales


def w8_gemm_workspace_size(M: int, K: int, N: int) -> int:
    return _size("qmm_w8_gemm_workspace_size", M, K, N)


def w8_gemm(codes: torch.Tensor, scales: torch.Tensor, N: int, K: int, X: torch.Tensor, Y=None, workspace=None,
            dev_status=None):
    """Y[m][n] = sum_b scales[n][b] sum_{k in b} codes[n][k] X[m][k]; X bf16 [M][K] on the device."""
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    if workspace is None:
        need = w8_gemm_workspace_size(M, K, N)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    _check("qmm_w8_gemm", lib.qmm_w8_gemm(
        _ptr(codes), _ptr(scales), N, K, _ptr(X), M, X.stride(0), _ptr(Y), Y.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream()))
    return Y


# ---------------------------------------------------------------------------
# More weight formats: Q4_K -> q4_1 tiles, Q8 tiles
# ---------------------------------------------------------------------------

def repack_q4k(q4k: torch.Tensor, N: int, K: int, tiles=None) -> torch.Tensor:
    """q4k: device uint8 [N][row_bytes] of Q4_K super-blocks (row_bytes >= K/256*144).
    Returns q4_1 tile bytes (uint8) for qmm_q4_gemm / qmm_q4_gemm_id."""
    nbytes = pack_q4_size(N, K)
    if tiles is None:
        tiles = torch.empty(nbytes, dtype=torch.uint8, device=q4k.device)
    row_bytes = q4k.stride(0) if q4k.dim() == 2 else K // 256 * 144
    _check("qmm_repack_q4k", lib.qmm_repack_q4k(_ptr(q4k), N, K, row_bytes, _ptr(tiles),
                                                tiles.numel(), _stream()))
    return tiles


def pack_q8_size(N: int, K: int) -> int:
    return _size("qmm_pack_q8_size", N, K)


def pack_q8(W: torch.Tensor, layout: int) -> torch.Tensor:
    """W: device fp32 [N][K].  Returns Q8 tile bytes (uint8) in the given code layout."""
    N, K = W.shape
    nbytes = pack_q8_size(N, K)
    tiles = torch.empty(nbytes, dtype=torch.uint8, device=W.device)
    _check("qmm_pack_q8", lib.qmm_pack_q8(_ptr(W), N, K, W.stride(0), int(layout), _ptr(tiles), nbytes,
                                          _stream()))
    return tiles


def q8_gemm_workspace_size(M: int, K: int, N: int) -> int:
    return _size("qmm_q8_gemm_workspace_size", M, K, N)


def q8_gemm(tiles: torch.Tensor, layout: int, N: int, K: int, X: torch.Tensor, Y=None, workspace=None,
            dev_status=None):
    """Y[m][n] = sum_k X[m][k] w[n][k] over Q8 tiles; X bf16 [M][K] on the device."""
    M = X.shape[0]
    if Y is None:
        Y = torch.empty((M, N), dtype=torch.float32, device=X.device)
    if workspace is None:
        need = q8_gemm_workspace_size(M, K, N)
        if need > 0:
            workspace = torch.empty(need, dtype=torch.uint8, device=X.device)
    _check("qmm_q8_gemm", lib.qmm_q8_gemm(
        _ptr(tiles), int(layout), N, K, _ptr(X), M, X.stride(0), _ptr(Y), Y.stride(0), _ptr(workspace),
        0 if workspace is None else workspace.numel() * workspace.element_size(), _ptr(dev_status), _stream()))
    return Y


# ---------------------------------------------------------------------------
# Diagnostics
# ---------------------------------------------------------------------------

def selftest_wait_timeout(limit_ns: int, dev_status: torch.Tensor, out: torch.Tensor):
    """Run the bounded-wait error path on purpose (see qmm_selftest_wait_timeout):
    dev_status (device int32 [1], zeroed by the caller) receives QMM_ERR_TIMEOUT
    and out (device int64 [4]) the wait results and times."""
    _check("qmm_selftest_wait_timeout", lib.qmm_selftest_wait_timeout(int(limit_ns), _ptr(dev_status), _ptr(out),
                                                                      _stream()))
    return out


def probe_hbm_read(buf: torch.Tensor, mode: int, sink: torch.Tensor, dev_status=None):
    """Load-only read of the whole of `buf` (see qmm_probe_hbm_read); sink is a
    device int32/uint32 [1] that normally stays untouched."""
    nbytes = buf.numel() * buf.element_size()
    _check("qmm_probe_hbm_read", lib.qmm_probe_hbm_read(_ptr(buf), nbytes, int(mode), _ptr(sink),
                                                        _ptr(dev_status), _stream()))
