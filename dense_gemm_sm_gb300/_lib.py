"""ctypes binding of libdgemm_sm103a.so -- argument marshalling only.

Every function keeps the C name and argument order of include/dgemm.h.  Matrix
arguments may be torch tensors (their data_ptr() is passed) or raw device
addresses (int).  `stream` defaults to torch's current CUDA stream.  A non-OK
status raises DgError unless check=False.  Nothing here computes: if the
shared library is missing this module raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

DG_OK, DG_ERR_INVALID_ARG, DG_ERR_MISALIGNED, DG_ERR_UNSUPPORTED = 0, 1, 2, 3
DG_ERR_CUDA, DG_ERR_TIMEOUT, DG_ERR_NO_MEMORY = 4, 5, 6
DG_OP_N, DG_OP_T = 0, 1
DG_OUT_BF16, DG_OUT_F32 = 0, 1
(DG_KERNEL_NONE, DG_KERNEL_SCALE, DG_KERNEL_SIMT_F32, DG_KERNEL_TC_BF16, DG_KERNEL_THIN_BF16,
 DG_KERNEL_TC2_BF16) = range(6)

EXPORTED = [
    "gemm_f32", "gemm_f32_strided_batched", "gemm_bf16", "gemm_bf16_strided_batched",
    "dg_status_string", "dg_device_status", "dg_release_workspace", "dg_plan_gemm",
    "dg_raster_tile", "dg_streamk_start", "dg_model_traffic_bytes", "dg_model_local_bytes",
    "dg_version", "dg_set_fault_injection", "gemm_bf16_decode_noalloc", "gemm_bf16_gate_up_silu",
    "attention_bf16", "quantize_rows_e4m3", "gemm_fp8_e4m3", "dg_model_quant_traffic_bytes",
    "gemm_bf16_decode_chain",
]


class DgError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {status_string(status)}")


class dg_plan(ctypes.Structure):
    _fields_ = [
        ("kernel", ctypes.c_int32), ("tile_m", ctypes.c_int32), ("tile_n", ctypes.c_int32),
        ("tile_k", ctypes.c_int32), ("stages", ctypes.c_int32), ("group", ctypes.c_int32),
        ("ntok", ctypes.c_int32), ("vec", ctypes.c_int32), ("splits", ctypes.c_int32),
        ("tiles", ctypes.c_int64), ("tail_tiles", ctypes.c_int64),
        ("grid", ctypes.c_int64), ("kblocks", ctypes.c_int64),
        ("workspace_bytes", ctypes.c_int64),
    ]

    def as_dict(self):
        return {name: getattr(self, name) for name, _ in self._fields_}


_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load(build_if_missing: bool = True):
    """Loads the shared library (building it first if it is absent or stale)."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB_PATH
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run dense_gemm_sm_gb300.build.build() first")
    lib = ctypes.CDLL(path)
    i64, i32, f32, vp = ctypes.c_int64, ctypes.c_int32, ctypes.c_float, ctypes.c_void_p
    lib.gemm_f32.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, vp]
    lib.gemm_f32_strided_batched.argtypes = [i64, i64, i64, f32, vp, i64, i64, vp, i64, i64, i32,
                                             f32, vp, i64, i64, i64, vp]
    lib.gemm_bf16.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64, i32, vp]
    lib.gemm_bf16_strided_batched.argtypes = [i64, i64, i64, f32, vp, i64, i64, vp, i64, i64, i32,
                                              f32, vp, i64, i64, i64, i32, vp]
    lib.gemm_bf16_gate_up_silu.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64, vp, i64, vp]
    lib.gemm_bf16_decode_chain.argtypes = [i32, i64, vp, vp, i64, vp, vp, vp, vp]
    lib.quantize_rows_e4m3.argtypes = [i64, i64, vp, i64, vp, i64, vp, vp]
    lib.gemm_fp8_e4m3.argtypes = [i64, i64, i64, vp, i64, vp, vp, i64, vp, vp, i64, i32, vp]
    lib.attention_bf16.argtypes = [i64, i64, i64, i64, f32, i32, vp, i64, i64, vp, i64, i64, vp,
                                   i64, i64, vp, i64, i64, vp]
    lib.gemm_bf16_decode_noalloc.argtypes = [i64, i64, i64, f32, vp, i64, vp, i64, f32, vp, i64,
                                             i32, vp]
    for f in ("gemm_f32", "gemm_f32_strided_batched", "gemm_bf16", "gemm_bf16_strided_batched",
              "gemm_bf16_decode_noalloc", "gemm_bf16_gate_up_silu", "attention_bf16",
              "quantize_rows_e4m3", "gemm_fp8_e4m3", "gemm_bf16_decode_chain"):
        getattr(lib, f).restype = ctypes.c_int
    lib.dg_status_string.argtypes = [ctypes.c_int]
    lib.dg_status_string.restype = ctypes.c_char_p
    lib.dg_device_status.argtypes = [vp]
    lib.dg_device_status.restype = ctypes.c_int
    lib.dg_release_workspace.argtypes = []
    lib.dg_release_workspace.restype = ctypes.c_int
    lib.dg_plan_gemm.argtypes = [i32, i64, i64, i64, i64, i32, i32, i32, ctypes.POINTER(dg_plan)]
    lib.dg_plan_gemm.restype = ctypes.c_int
    p64 = ctypes.POINTER(ctypes.c_int64)
    lib.dg_raster_tile.argtypes = [i64, i64, i64, i32, p64, p64, p64]
    lib.dg_raster_tile.restype = None
    lib.dg_streamk_start.argtypes = [i64, i64, i64]
    lib.dg_streamk_start.restype = i64
    lib.dg_model_traffic_bytes.argtypes = [i64, i64, i64, i64, i64, i32, i32]
    lib.dg_model_traffic_bytes.restype = ctypes.c_double
    lib.dg_model_local_bytes.argtypes = [i64, i64, i64, i32]
    lib.dg_model_local_bytes.restype = i64
    lib.dg_model_quant_traffic_bytes.argtypes = [i64, i64, i64, i64, i64, i32, i32, i32, i32]
    lib.dg_model_quant_traffic_bytes.restype = ctypes.c_double
    lib.dg_version.argtypes = []
    lib.dg_version.restype = ctypes.c_char_p
    lib.dg_set_fault_injection.argtypes = [i32]
    lib.dg_set_fault_injection.restype = None
    _lib = lib
    return lib


def _ptr(x) -> int:
    if x is None:
        return 0
    if hasattr(x, "data_ptr"):
        return int(x.data_ptr())
    return int(x)


def _stream(stream) -> int:
    if stream is None:
        import torch
        if torch.cuda.is_available():
            return int(torch.cuda.current_stream().cuda_stream)
        return 0
    if hasattr(stream, "cuda_stream"):
        return int(stream.cuda_stream)
    return int(stream)


def _ret(status: int, where: str, check: bool) -> int:
    if check and status != DG_OK:
        raise DgError(status, where)
    return status


def gemm_f32(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, stream=None, check=True) -> int:
    lib = load()
    st = lib.gemm_f32(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc,
                      _stream(stream))
    return _ret(st, "gemm_f32", check)


def gemm_f32_strided_batched(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, op_b, beta, C, ldc,
                             strideC, batch, stream=None, check=True) -> int:
    lib = load()
    st = lib.gemm_f32_strided_batched(M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb, strideB,
                                      op_b, beta, _ptr(C), ldc, strideC, batch, _stream(stream))
    return _ret(st, "gemm_f32_strided_batched", check)


def gemm_bf16(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type=DG_OUT_BF16, stream=None,
              check=True) -> int:
    lib = load()
    st = lib.gemm_bf16(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C), ldc, c_type,
                       _stream(stream))
    return _ret(st, "gemm_bf16", check)


def gemm_bf16_strided_batched(M, N, K, alpha, A, lda, strideA, B, ldb, strideB, op_b, beta, C, ldc,
                              strideC, batch, c_type=DG_OUT_BF16, stream=None, check=True) -> int:
    lib = load()
    st = lib.gemm_bf16_strided_batched(M, N, K, alpha, _ptr(A), lda, strideA, _ptr(B), ldb,
                                       strideB, op_b, beta, _ptr(C), ldc, strideC, batch, c_type,
                                       _stream(stream))
    return _ret(st, "gemm_bf16_strided_batched", check)


def gemm_bf16_decode_noalloc(M, N, K, alpha, A, lda, B, ldb, beta, C, ldc, c_type=DG_OUT_BF16,
                             stream=None, check=True) -> int:
    """Decode-shaped gemm_bf16 (M <= 16) that allocates nothing (fixed scratch in the library)."""
    lib = load()
    st = lib.gemm_bf16_decode_noalloc(M, N, K, alpha, _ptr(A), lda, _ptr(B), ldb, beta, _ptr(C),
                                      ldc, c_type, _stream(stream))
    return _ret(st, "gemm_bf16_decode_noalloc", check)


def gemm_bf16_gate_up_silu(M, N, K, X, ldx, Wg, ldwg, Wu, ldwu, Z, ldz, stream=None,
                           check=True) -> int:
    """Z = bf16(SiLU(bf16(X Wg)) * bf16(X Wu)): FFN gate/up projections, activation fused."""
    lib = load()
    st = lib.gemm_bf16_gate_up_silu(M, N, K, _ptr(X), ldx, _ptr(Wg), ldwg, _ptr(Wu), ldwu,
                                    _ptr(Z), ldz, _stream(stream))
    return _ret(st, "gemm_bf16_gate_up_silu", check)


def gemm_bf16_decode_chain(M, dims, X, ldx, Ws, ldws, Ys, stream=None, check=True) -> int:
    """Y[0] = bf16(X W[0]), Y[l] = bf16(Y[l-1] W[l]): `len(Ws)` decode GEMMs in one launch."""
    lib = load()
    layers = len(Ws)
    dims_a = (ctypes.c_int64 * (layers + 1))(*[int(d) for d in dims])
    ldw_a = (ctypes.c_int64 * layers)(*[int(v) for v in ldws])
    w_a = (ctypes.c_void_p * layers)(*[_ptr(w) for w in Ws])
    y_a = (ctypes.c_void_p * layers)(*[_ptr(y) for y in Ys])
    st = lib.gemm_bf16_decode_chain(layers, M, ctypes.cast(dims_a, ctypes.c_void_p), _ptr(X), ldx,
                                    ctypes.cast(w_a, ctypes.c_void_p), ctypes.cast(ldw_a, ctypes.c_void_p),
                                    ctypes.cast(y_a, ctypes.c_void_p), _stream(stream))
    return _ret(st, "gemm_bf16_decode_chain", check)


def quantize_rows_e4m3(rows, cols, X, ldx, Q, ldq, scales, stream=None, check=True) -> int:
    """Per-row FP8 E4M3 quantisation of BF16 X: codes Q and float32 scales (amax / 448)."""
    lib = load()
    st = lib.quantize_rows_e4m3(rows, cols, _ptr(X), ldx, _ptr(Q), ldq, _ptr(scales),
                                _stream(stream))
    return _ret(st, "quantize_rows_e4m3", check)


def gemm_fp8_e4m3(M, N, K, A, lda, scale_a, B, ldb, scale_b, C, ldc, c_type=DG_OUT_BF16,
                  stream=None, check=True) -> int:
    """C = diag(scale_a) (A B^T) diag(scale_b) for E4M3 codes A [M, K] and B [N, K]."""
    lib = load()
    st = lib.gemm_fp8_e4m3(M, N, K, _ptr(A), lda, _ptr(scale_a), _ptr(B), ldb, _ptr(scale_b),
                           _ptr(C), ldc, c_type, _stream(stream))
    return _ret(st, "gemm_fp8_e4m3", check)


def attention_bf16(batch, Lq, Lkv, d, scale, causal, Q, ldq, strideQ, K, ldk, strideK, V, ldv,
                   strideV, O, ldo, strideO, stream=None, check=True) -> int:
    """O = softmax(scale * Q K^T) V per head (fused, online softmax), BF16 in and out."""
    lib = load()
    st = lib.attention_bf16(batch, Lq, Lkv, d, scale, 1 if causal else 0, _ptr(Q), ldq, strideQ,
                            _ptr(K), ldk, strideK, _ptr(V), ldv, strideV, _ptr(O), ldo, strideO,
                            _stream(stream))
    return _ret(st, "attention_bf16", check)


def status_string(status: int) -> str:
    return load().dg_status_string(status).decode()


dg_status_string = status_string


def dg_device_status(stream=None) -> int:
    return load().dg_device_status(_stream(stream))


def dg_release_workspace() -> int:
    return load().dg_release_workspace()


def dg_plan_gemm(dtype, M, N, K, batch=1, op_b=DG_OP_N, c_type=DG_OUT_BF16, num_sms=0) -> dict:
    out = dg_plan()
    st = load().dg_plan_gemm(dtype, M, N, K, batch, op_b, c_type, num_sms, ctypes.byref(out))
    _ret(st, "dg_plan_gemm", True)
    return out.as_dict()


def dg_raster_tile(t, tiles_m, tiles_n, group):
    b, tm, tn = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
    load().dg_raster_tile(t, tiles_m, tiles_n, group, ctypes.byref(b), ctypes.byref(tm),
                          ctypes.byref(tn))
    return b.value, tm.value, tn.value


def dg_streamk_start(c, units, ctas) -> int:
    return load().dg_streamk_start(c, units, ctas)


def dg_model_traffic_bytes(M, N, K, tile_m, tile_n, elem_bytes=2, out_bytes=2) -> float:
    return load().dg_model_traffic_bytes(M, N, K, tile_m, tile_n, elem_bytes, out_bytes)


def dg_model_local_bytes(tile_m, tile_n, tile_k, elem_bytes=2) -> int:
    return load().dg_model_local_bytes(tile_m, tile_n, tile_k, elem_bytes)


def dg_model_quant_traffic_bytes(M, K, N, tile_m, tile_n, in_bytes=2, q_bytes=1, out_bytes=2,
                                 fused=False) -> float:
    return load().dg_model_quant_traffic_bytes(M, K, N, tile_m, tile_n, in_bytes, q_bytes,
                                               out_bytes, 1 if fused else 0)


def dg_version() -> str:
    return load().dg_version().decode()


def dg_set_fault_injection(mode: int) -> None:
    load().dg_set_fault_injection(mode)
