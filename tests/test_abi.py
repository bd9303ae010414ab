"""CPU tests of the C ABI: the library loads, exports every declared symbol,
and rejects bad arguments on the host before touching the GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "qmm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qmm_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(qmm):
    names = declared_functions()
    assert len(names) >= 11
    lib = ctypes.CDLL(qmm.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) <= set(qmm.SIGNATURES)


def test_status_strings(qmm):
    assert qmm.status_string(0) == "QMM_OK"
    assert qmm.status_string(6) == "QMM_ERR_BAD_EXPERT_ID"
    assert qmm.status_string(8) == "QMM_ERR_RANGE"
    assert qmm.status_string(99) == "QMM_ERR_UNKNOWN"


def test_size_queries(qmm):
    assert qmm.pack_b_int8_size(1, 1) == 64
    assert qmm.pack_b_int8_size(1024, 3) == 3 * 1024
    assert qmm.pack_b_int8_size(1025, 3) == 3 * 1088
    assert qmm.pack_q4_size(32, 256) == 5120
    assert qmm.pack_q4_size(151936, 1024) == 97239040
    assert qmm.int8_gemm_workspace_size(16, 1024, 1024) >= 0
    # MUL_MAT_ID: routing tables and row scales (256-byte padded) + packed f16 activation rows
    assert qmm.q4_gemm_id_workspace_size(128, 8, 512, 2048) == 768 + 16384 + 16384 + 4096 * 2048 * 2
    # dense q4: nothing for the decode GEMV; f16 activation rows + row scales for the tensor-core route
    assert qmm.q4_gemm_workspace_size(16, 1024, 64) == 0
    assert qmm.q4_gemm_workspace_size(17, 1024, 64) == 17 * 1024 * 2 + 256
    assert qmm.q4_gemm_workspace_size(300, 2048, 96) == 300 * 2048 * 2 + 1280
    L = qmm.lib
    sz = ctypes.c_size_t(0)
    assert L.qmm_q4_gemm_id_workspace_size(128, 8, 512, 300, ctypes.byref(sz)) == qmm.QMM_ERR_UNSUPPORTED


def test_overflow_bound_rejected(qmm):
    # int8 inference, "Product kernel": safe while K*255*128 < 2^31
    kmax = (2 ** 31 - 1) // (255 * 128)
    assert qmm.pack_b_int8_size(kmax, 1) > 0
    with pytest.raises(qmm.QmmError) as e:
        qmm.pack_b_int8_size(kmax + 1, 1)
    assert e.value.status == qmm.QMM_ERR_OVERFLOW_BOUND


def test_q4_unsupported_shapes(qmm):
    for N, K in ((33, 256), (32, 255), (64, 300)):
        with pytest.raises(qmm.QmmError) as e:
            qmm.pack_q4_size(N, K)
        assert e.value.status == qmm.QMM_ERR_UNSUPPORTED


def _call(qmm, name, *args):
    return getattr(qmm.lib, name)(*args)


def test_host_validation_before_launch(qmm):
    L = qmm.lib
    P = ctypes.c_void_p(1 << 20)      # aligned fake device address: never dereferenced
    U = ctypes.c_void_p((1 << 20) + 3)  # misaligned
    ep = qmm.QmmEpilogue(qmm.QMM_S32, None, None, 0, None, 1.0, 0)
    epb = ctypes.byref(ep)
    g = lambda *a: L.qmm_int8_gemm(*a)
    # null A
    assert g(None, qmm.QMM_U8, 4, 16, 16, 0, P, P, 8, qmm.QMM_S8, 0, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    # misaligned A, lda not a multiple of 16
    assert g(U, qmm.QMM_U8, 4, 16, 16, 0, P, P, 8, qmm.QMM_S8, 0, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, qmm.QMM_U8, 4, 16, 24, 0, P, P, 8, qmm.QMM_S8, 0, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    # zero point outside the operand domain; zB != 0 for fp32 weights
    assert g(P, qmm.QMM_U8, 4, 16, 16, 256, P, P, 8, qmm.QMM_S8, 0, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, qmm.QMM_S8, 4, 16, 16, 0, P, P, 8, qmm.QMM_S8, 200, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, qmm.QMM_S8, 4, 16, 16, 0, P, P, 8, qmm.QMM_F32, 1, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    # K beyond the int32 bound
    assert g(P, qmm.QMM_S8, 4, 70000, 70000, 0, P, P, 8, qmm.QMM_S8, 0, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_OVERFLOW_BOUND
    # ldo < N, bad output type, requant without a positive s_y
    assert g(P, qmm.QMM_S8, 4, 16, 16, 0, P, P, 8, qmm.QMM_S8, 0, epb, P, 7, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    bad = qmm.QmmEpilogue(qmm.QMM_BF16, None, None, 0, None, 1.0, 0)
    assert g(P, qmm.QMM_S8, 4, 16, 16, 0, P, P, 8, qmm.QMM_S8, 0, ctypes.byref(bad), P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    rq = qmm.QmmEpilogue(qmm.QMM_S8, None, None, 0, None, 0.0, 0)
    assert g(P, qmm.QMM_S8, 4, 16, 16, 0, P, P, 8, qmm.QMM_S8, 0, ctypes.byref(rq), P, 8, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    # q4: shapes off the tile grid, X row stride not a multiple of 8
    assert L.qmm_q4_gemm(P, 33, 256, P, 1, 256, P, 33, None, 0, None, None) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_q4_gemm(P, 32, 256, P, 1, 260, P, 32, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    # q4 tensor-core route (M >= 17): missing, short or misaligned workspace
    assert L.qmm_q4_gemm(P, 32, 256, P, 17, 256, P, 32, None, 0, None, None) == qmm.QMM_ERR_WORKSPACE
    assert L.qmm_q4_gemm(P, 32, 256, P, 17, 256, P, 32, P, 17 * 256 * 2, None, None) == qmm.QMM_ERR_WORKSPACE
    assert L.qmm_q4_gemm(P, 32, 256, P, 17, 256, P, 32, ctypes.c_void_p((1 << 20) + 128), 1 << 20, None,
                         None) == qmm.QMM_ERR_WORKSPACE
    # MUL_MAT_ID: ld_ids < n_used, missing workspace
    assert L.qmm_q4_gemm_id(P, 4, 32, 256, P, 256, 0, P, 2, 3, 5, P, 96, 32, P, 1 << 20, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_q4_gemm_id(P, 4, 32, 256, P, 256, 0, P, 17, 3, 5, P, 96, 32, None, 0, None, None) == qmm.QMM_ERR_WORKSPACE
    # pack: fp32 weights need a scale output
    assert L.qmm_pack_b_int8(P, qmm.QMM_F32, 16, 8, 8, P, 1 << 20, None, P, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_pack_q4(P, 32, 256, 100, P, 5120, None) == qmm.QMM_ERR_INVALID_ARG


def test_binding_has_no_oracle_imports():
    # the product path never imports the oracle
    for f in ("qmm.py", "build.py", "__init__.py", "inputs.py"):
        src = open(os.path.join(ROOT, "quantized_matmul_qmm_gb300", f)).read()
        assert not re.search(r"^\s*(import|from)\s+oracle", src, flags=re.M), f


def test_quantize_act_host_validation(qmm):
    L = qmm.lib
    P = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: every call below fails on the host
    sz = ctypes.c_size_t(0)
    assert L.qmm_quantize_act_int8_workspace_size(4, 16, 0, ctypes.byref(sz)) == qmm.QMM_OK and sz.value == 256
    assert L.qmm_quantize_act_int8_workspace_size(4, 16, 1, ctypes.byref(sz)) == qmm.QMM_OK and sz.value == 0
    assert L.qmm_quantize_act_int8_workspace_size(4, 16, 2, ctypes.byref(sz)) == qmm.QMM_ERR_INVALID_ARG
    q = L.qmm_quantize_act_int8
    # x_type, per_row, lda % 16, lda < K, ldx < K, misaligned A, missing per-tensor workspace
    assert q(P, qmm.QMM_S8, 4, 16, 16, 1, P, 16, P, None, 0, None) == qmm.QMM_ERR_INVALID_ARG
    assert q(P, qmm.QMM_F32, 4, 16, 16, 2, P, 16, P, None, 0, None) == qmm.QMM_ERR_INVALID_ARG
    assert q(P, qmm.QMM_F32, 4, 16, 16, 1, P, 24, P, None, 0, None) == qmm.QMM_ERR_INVALID_ARG
    assert q(P, qmm.QMM_F32, 4, 40, 40, 1, P, 32, P, None, 0, None) == qmm.QMM_ERR_INVALID_ARG
    assert q(P, qmm.QMM_F32, 4, 40, 39, 1, P, 48, P, None, 0, None) == qmm.QMM_ERR_INVALID_ARG
    assert q(P, qmm.QMM_F32, 4, 16, 16, 1, ctypes.c_void_p((1 << 20) + 8), 16, P, None, 0, None) == qmm.QMM_ERR_INVALID_ARG
    assert q(P, qmm.QMM_F32, 4, 16, 16, 0, P, 16, P, None, 0, None) == qmm.QMM_ERR_WORKSPACE
    assert q(P, qmm.QMM_F32, 4, 16, 16, 0, P, 16, P, P, 64, None) == qmm.QMM_ERR_WORKSPACE


def test_w8_sizes_and_host_validation(qmm):
    # codes N x Kp (K rounded up to 64), scales N x ceil(K / 1024) fp32
    assert qmm.pack_w8_size(3, 1) == (3 * 64, 3 * 4)
    assert qmm.pack_w8_size(1024, 1024) == (1024 * 1024, 1024 * 4)
    assert qmm.pack_w8_size(7, 1025) == (7 * 1088, 7 * 2 * 4)
    assert qmm.pack_w8_size(2, 65536) == (2 * 65536, 2 * 64 * 4)
    assert qmm.w8_gemm_workspace_size(16, 1000, 300) == 0
    assert qmm.w8_gemm_workspace_size(17, 1000, 300) == 300 * 1024 * 2
    L = qmm.lib
    P = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: every call below fails on the host
    cb, sb = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.qmm_pack_w8_size(2, 65537, ctypes.byref(cb), ctypes.byref(sb)) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_pack_w8_size(0, 16, ctypes.byref(cb), ctypes.byref(sb)) == qmm.QMM_ERR_INVALID_ARG
    pk = L.qmm_pack_w8
    # ldw < K, short code buffer, short scale buffer, misaligned codes
    assert pk(P, 4, 100, 99, P, 4 * 128, P, 16, None) == qmm.QMM_ERR_INVALID_ARG
    assert pk(P, 4, 100, 100, P, 4 * 128 - 1, P, 16, None) == qmm.QMM_ERR_INVALID_ARG
    assert pk(P, 4, 100, 100, P, 4 * 128, P, 15, None) == qmm.QMM_ERR_INVALID_ARG
    assert pk(P, 4, 100, 100, ctypes.c_void_p((1 << 20) + 8), 4 * 128, P, 16, None) == qmm.QMM_ERR_INVALID_ARG
    g = L.qmm_w8_gemm
    # ldx % 8, ldx < K, ldy < N, misaligned X, K too large, missing or short workspace (M > 16)
    assert g(P, P, 64, 100, P, 4, 100, P, 64, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, P, 64, 100, P, 4, 96, P, 64, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, P, 64, 96, P, 4, 96, P, 63, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, P, 64, 96, ctypes.c_void_p((1 << 20) + 2), 4, 96, P, 64, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, P, 64, 65544, P, 4, 65544, P, 64, None, 0, None, None) == qmm.QMM_ERR_UNSUPPORTED
    assert g(P, P, 64, 96, P, 17, 96, P, 64, None, 0, None, None) == qmm.QMM_ERR_WORKSPACE
    assert g(P, P, 64, 96, P, 17, 96, P, 64, P, 64 * 128 * 2 - 1, None, None) == qmm.QMM_ERR_WORKSPACE


def test_format_sizes_and_host_validation(qmm):
    # Q8 tiles: 8192 code bytes + 512 scale bytes per 32 x 256 tile
    assert qmm.pack_q8_size(32, 256) == 8704
    assert qmm.pack_q8_size(151936, 1024) == 4748 * 4 * 8704
    assert qmm.q8_gemm_workspace_size(16, 1024, 64) == 0
    # f16 weights, chunk scales, f16 activation rows, row scales (each rounded up to 256)
    assert qmm.q8_gemm_workspace_size(17, 1024, 64) == 64 * 1024 * 2 + 256 + 17 * 1024 * 2 + 256
    assert qmm.q8_gemm_workspace_size(17, 2048, 96) == 96 * 2048 * 2 + 768 + 17 * 2048 * 2 + 256
    L = qmm.lib
    P = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: every call below fails on the host
    sz = ctypes.c_size_t(0)
    assert L.qmm_pack_q8_size(33, 256, ctypes.byref(sz)) == qmm.QMM_ERR_UNSUPPORTED
    assert L.qmm_q8_gemm_workspace_size(17, 65792, 32, ctypes.byref(sz)) == qmm.QMM_ERR_UNSUPPORTED
    # repack: off the tile grid, short row stride, row stride not a multiple of 16, short tiles, misaligned
    rp = L.qmm_repack_q4k
    assert rp(P, 33, 256, 144, P, 1 << 20, None) == qmm.QMM_ERR_UNSUPPORTED
    assert rp(P, 32, 512, 272, P, 1 << 20, None) == qmm.QMM_ERR_INVALID_ARG
    assert rp(P, 32, 256, 152, P, 1 << 20, None) == qmm.QMM_ERR_INVALID_ARG
    assert rp(P, 32, 256, 144, P, 5119, None) == qmm.QMM_ERR_INVALID_ARG
    assert rp(ctypes.c_void_p((1 << 20) + 8), 32, 256, 144, P, 5120, None) == qmm.QMM_ERR_INVALID_ARG
    # pack_q8: bad layout, ldw < K, short tiles
    pk = L.qmm_pack_q8
    assert pk(P, 32, 256, 256, 2, P, 8704, None) == qmm.QMM_ERR_INVALID_ARG
    assert pk(P, 32, 256, 255, 0, P, 8704, None) == qmm.QMM_ERR_INVALID_ARG
    assert pk(P, 32, 256, 256, 1, P, 8703, None) == qmm.QMM_ERR_INVALID_ARG
    g = L.qmm_q8_gemm
    # bad layout, off the grid, ldx % 8, misaligned X, missing or short workspace (M > 16), K too large
    assert g(P, 5, 32, 256, P, 1, 256, P, 32, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, 0, 48, 256, P, 1, 256, P, 48, None, 0, None, None) == qmm.QMM_ERR_UNSUPPORTED
    assert g(P, 0, 32, 256, P, 1, 260, P, 32, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, 0, 32, 256, ctypes.c_void_p((1 << 20) + 2), 1, 256, P, 32, None, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, 1, 32, 256, P, 17, 256, P, 32, None, 0, None, None) == qmm.QMM_ERR_WORKSPACE
    assert g(P, 1, 32, 256, P, 17, 256, P, 32, P, 32 * 256 * 2, None, None) == qmm.QMM_ERR_WORKSPACE
    assert g(P, 1, 32, 65792, P, 17, 65792, P, 32, P, 1 << 30, None, None) == qmm.QMM_ERR_UNSUPPORTED


def test_axis_zp_sizes_and_host_validation(qmm):
    # int32 product [M][N] + row sums [M] (each rounded up to 256) + the GEMM's own workspace
    assert qmm.int8_gemm_axis_zp_workspace_size(16, 1024, 1024) == 16 * 1024 * 4 + 256 + \
        qmm.int8_gemm_workspace_size(16, 1024, 1024)
    assert qmm.int8_gemm_axis_zp_workspace_size(300, 64, 7) == 8448 + 1280 + qmm.int8_gemm_workspace_size(300, 64, 7)
    L = qmm.lib
    P = ctypes.c_void_p(1 << 20)   # aligned, never dereferenced: every call below fails on the host
    ep = qmm.QmmEpilogue(qmm.QMM_S32, None, None, 0, None, 1.0, 0)
    epb = ctypes.byref(ep)
    g = L.qmm_int8_gemm_axis_zp
    big = 1 << 30
    # column zero points with fp32 (symmetric) weights; misaligned zero points; missing workspace;
    # K beyond the int32 bound; bad output type
    assert g(P, qmm.QMM_S8, 4, 16, 16, None, P, P, 8, qmm.QMM_F32, P, epb, P, 8, P, big, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, qmm.QMM_S8, 4, 16, 16, ctypes.c_void_p((1 << 20) + 2), P, P, 8, qmm.QMM_S8, P, epb, P, 8, P, big,
             None, None) == qmm.QMM_ERR_INVALID_ARG
    assert g(P, qmm.QMM_S8, 4, 16, 16, P, P, P, 8, qmm.QMM_S8, P, epb, P, 8, None, 0, None, None) == qmm.QMM_ERR_WORKSPACE
    assert g(P, qmm.QMM_S8, 4, 16, 16, P, P, P, 8, qmm.QMM_S8, P, epb, P, 8, P, 255, None, None) == qmm.QMM_ERR_WORKSPACE
    assert g(P, qmm.QMM_S8, 4, 70000, 70000, P, P, P, 8, qmm.QMM_S8, P, epb, P, 8, P, big, None, None) == qmm.QMM_ERR_OVERFLOW_BOUND
    bad = qmm.QmmEpilogue(qmm.QMM_BF16, None, None, 0, None, 1.0, 0)
    assert g(P, qmm.QMM_S8, 4, 16, 16, P, P, P, 8, qmm.QMM_S8, P, ctypes.byref(bad), P, 8, P, big, None,
             None) == qmm.QMM_ERR_INVALID_ARG


def test_q4_gemv_group_host_validation(qmm):
    """The grouped decode GEMV checks every descriptor on the host: a bad one
    fails the whole call before anything is queued."""
    L = qmm.lib
    P = 1 << 20   # aligned, never dereferenced
    Pr = qmm.QmmQ4GemvProblem
    good = Pr(P, 64, 512, P, P)

    def call(*probs):
        arr = (Pr * len(probs))(*probs)
        return L.qmm_q4_gemv_group(arr, len(probs), None, None)

    assert L.qmm_q4_gemv_group(None, 1, None, None) == qmm.QMM_ERR_INVALID_ARG
    arr = (Pr * 1)(good)
    assert L.qmm_q4_gemv_group(arr, 0, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert call(good, Pr(P, 48, 512, P, P)) == qmm.QMM_ERR_UNSUPPORTED        # N % 32
    assert call(good, Pr(P, 64, 500, P, P)) == qmm.QMM_ERR_UNSUPPORTED        # K % 256
    assert call(good, Pr(None, 64, 512, P, P)) == qmm.QMM_ERR_INVALID_ARG     # null tiles
    assert call(Pr(P, 64, 512, P + 8, P), good) == qmm.QMM_ERR_INVALID_ARG    # x not 16-byte aligned
    assert call(good, Pr(P, 64, 512, P, P + 2)) == qmm.QMM_ERR_INVALID_ARG    # y not 4-byte aligned
    assert call(good, Pr(P, 0, 512, P, P)) == qmm.QMM_ERR_INVALID_ARG         # empty problem


def test_int8_gemm_group_host_validation(qmm):
    """The grouped small-M int8 GEMM applies qmm_int8_gemm's host checks to
    every problem and refuses M > 64, before anything is queued."""
    L = qmm.lib
    P = 1 << 20
    ep = qmm.QmmEpilogue(qmm.QMM_S32, None, None, 0, None, 1.0, 0)

    def prob(M=16, K=64, lda=64, zA=128, N=32, a_type=qmm.QMM_U8, b_type=qmm.QMM_S8, zB=0, out=P, ldo=32):
        return qmm.QmmInt8Problem(P, a_type, M, K, lda, zA, P, P, N, b_type, zB, ep, out, ldo)

    def call(*probs):
        arr = (qmm.QmmInt8Problem * len(probs))(*probs)
        return L.qmm_int8_gemm_group(arr, len(probs), None, None)

    assert L.qmm_int8_gemm_group(None, 1, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert call(prob(), prob(M=65)) == qmm.QMM_ERR_UNSUPPORTED            # beyond the small-M route
    assert call(prob(), prob(lda=72)) == qmm.QMM_ERR_INVALID_ARG          # lda % 16
    assert call(prob(zA=300)) == qmm.QMM_ERR_INVALID_ARG                  # zero point outside uint8
    assert call(prob(ldo=31)) == qmm.QMM_ERR_INVALID_ARG                  # ldo < N
    assert call(prob(K=70000, lda=70016)) == qmm.QMM_ERR_OVERFLOW_BOUND
    assert call(prob(out=P + 2)) == qmm.QMM_ERR_INVALID_ARG               # int32 output misaligned


def test_q4_gemm_id_pair_host_validation(qmm):
    L = qmm.lib
    P = ctypes.c_void_p(1 << 20)
    # a missing or misaligned second weight set / output, then the single call's checks
    assert L.qmm_q4_gemm_id_pair(P, None, 4, 32, 256, P, 256, P, 3, 2, 5, P, P, 64, 32, P, 1 << 20, None,
                                 None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_q4_gemm_id_pair(P, P, 4, 32, 256, P, 256, P, 3, 2, 5, P, None, 64, 32, P, 1 << 20, None,
                                 None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_q4_gemm_id_pair(P, ctypes.c_void_p((1 << 20) + 8), 4, 32, 256, P, 256, P, 3, 2, 5, P, P, 64, 32, P,
                                 1 << 20, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_q4_gemm_id_pair(P, P, 4, 32, 256, P, 256, P, 1, 2, 5, P, P, 64, 32, P, 1 << 20, None,
                                 None) == qmm.QMM_ERR_INVALID_ARG   # ld_ids < n_used
    assert L.qmm_q4_gemm_id_pair(P, P, 4, 32, 256, P, 256, P, 3, 2, 5, P, P, 64, 32, None, 0, None,
                                 None) == qmm.QMM_ERR_WORKSPACE


def test_widen_b_sizes_and_host_validation(qmm):
    """The one-time f16 copy of packed int8 weights and the GEMM that reads
    it: sizes, and bad arguments rejected on the host."""
    L = qmm.lib
    sz = ctypes.c_size_t(0)
    assert L.qmm_widen_b_int8_size(100, 7, ctypes.byref(sz)) == qmm.QMM_OK and sz.value == 7 * 128 * 2
    assert L.qmm_widen_b_int8_size(0, 7, ctypes.byref(sz)) == qmm.QMM_ERR_INVALID_ARG
    kmax = (2 ** 31 - 1) // (255 * 128)
    assert L.qmm_widen_b_int8_size(kmax + 1, 7, ctypes.byref(sz)) == qmm.QMM_ERR_OVERFLOW_BOUND
    # the b16 call needs less workspace: no room for the widened weights
    full, b16ws = ctypes.c_size_t(0), ctypes.c_size_t(0)
    assert L.qmm_int8_gemm_workspace_size(4096, 4608, 4608, ctypes.byref(full)) == qmm.QMM_OK
    assert L.qmm_int8_gemm_b16_workspace_size(4096, 4608, 4608, ctypes.byref(b16ws)) == qmm.QMM_OK
    assert full.value - b16ws.value >= 4608 * 4608 * 2
    assert L.qmm_int8_gemm_b16_workspace_size(16, 1024, 1024, ctypes.byref(b16ws)) == qmm.QMM_OK and b16ws.value == 0
    p16 = 1 << 20   # a 16-byte aligned, never dereferenced address
    assert L.qmm_widen_b_int8(None, 64, 8, p16, 1024, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_widen_b_int8(p16, 64, 8, None, 1024, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_widen_b_int8(p16 + 4, 64, 8, p16, 1024, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_widen_b_int8(p16, 64, 8, p16 + 8, 1024, None, None) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_widen_b_int8(p16, 64, 8, p16, 1023, None, None) == qmm.QMM_ERR_INVALID_ARG
    ep = qmm.QmmEpilogue(qmm.DTYPES["s32"], None, None, 0, None, 1.0, 0)
    args = lambda b16: (p16, qmm.DTYPES["u8"], 128, 64, 64, 0, p16, b16, p16, 8, qmm.DTYPES["s8"], 0,
                        ctypes.byref(ep), p16, 8, p16, 1 << 30, None, None)
    assert L.qmm_int8_gemm_b16(*args(None)) == qmm.QMM_ERR_INVALID_ARG
    assert L.qmm_int8_gemm_b16(*args(p16 + 2)) == qmm.QMM_ERR_INVALID_ARG
