"""ctypes binding of libnvfp4rac.so: argument marshalling only.

Every function here forwards torch tensors' device pointers and the current CUDA stream to the
C ABI declared in include/nvfp4rac.h and raises if the library returns an error.  There is no
fallback: if the library cannot be loaded the import of this module fails.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

from . import build as _build

_P, _I64, _I32, _U64 = C.c_void_p, C.c_int64, C.c_int32, C.c_uint64

_SIGS = {
    "nvq_last_error": ([], C.c_char_p),
    "nvq_device_status": ([_P, _P, _P], C.c_int),
    "nvq_set_wait_limit": ([_U64], C.c_int),
    "nvq_set_tail_path": ([_I32], C.c_int),
    "nvq_fp4_mma_rate": ([_I32, _I32, _P, _P], C.c_int),
    "nvq_sf_cols": ([_I64], _I64),
    "nvq_sf_bytes": ([_I64, _I64], _I64),
    "nvq_sf_offset": ([_I64, _I64, _I64], _I64),
    "nvfp4_quantize": ([_P, _I64, _I64, _I64, _P, _P, _I32, _P, _I64, _P, _I64, _I32, _P, _P, _I32, _P], C.c_int),
    "nvfp4_amax": ([_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P], C.c_int),
    "nvq_check_block_scale_division": ([_P, _P], C.c_int),
    "rac_select_quantize": ([_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _I32, _P, _I64, _P, _I64, _P, _P], C.c_int),
    "weight_qdq": ([_P, _I32, _I64, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _I32, _P], C.c_int),
    "w4a4_rac_grouped_gemm": ([_I32, _P, _P, _I64, _P, _I64, _P, _I64, _P, _I32, _P, _I64, _P, _I64, _P, _I64, _I64,
                               _I32, _P, _I32, _I32, _P, _P, _I64, _P, _P], C.c_int),
    "rac_select": ([_P, _I64, _I32, _I32, _P, _P], C.c_int),
    "rac_residual_tail": ([_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _I32, _P, _I64, _P, _I64, _P], C.c_int),
    "rac_reconstruct": ([_P, _I64, _P, _I64, _P, _I64, _I64, _I32, _P, _P, _P, _I32, _P, _I64, _P], C.c_int),
    "rac_weight_tail": ([_I32, _I64, _I64, _I32, _P, _I32, _P, _I64, _P, _I64, _P, _P, _P, _P], C.c_int),
    "nvfp4_channel_major": ([_I32, _I64, _I64, _P, _I64, _P, _I64, _P, _P, _P], C.c_int),
    "moe_capacity": ([_I64, _I32, _I32], _I64),
    "moe_dispatch_workspace_size": ([_I64, _I32, _I32], C.c_size_t),
    "moe_dispatch": ([_P, _P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _I64, _P, C.c_size_t, _P], C.c_int),
    "moe_dispatch_static_scratch": ([_P, _P, _I64, _I32, _I32, _P, _P, _P, _P, _P, _I64, _P], C.c_int),
    "nvfp4_gather_rows": ([_P, _I64, _P, _I64, _I64, _P, _I32, _I64, _I64, _I64, _P, _I64, _P, _P], C.c_int),
    "nvq_fp8_sf_cols": ([_I64], _I64),
    "fp8_quantize": ([_P, _I64, _I64, _I64, _I32, _P, _I64, _P, _I64, _P], C.c_int),
    "fp8_blockscaled_grouped_gemm": ([_I32, _P, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _P, _I64, _I64, _I64, _I32, _P, _P,
                                      _I64, _P], C.c_int),
    "fp8_gather_rows": ([_P, _I64, _P, _I64, _I64, _P, _I32, _I64, _I64, _P, _I64, _P, _P], C.c_int),
    "moe_combine": ([_P, _I64, _P, _I64, _I32, _I64, _P, _I64, _P], C.c_int),
}

EXPORTED = tuple(_SIGS)

NVQ_EPI_STORE, NVQ_EPI_SWIGLU, NVQ_EPI_ROW_SCALE, NVQ_EPI_STORE_F32 = 0, 1, 2, 3
NVQ_BF16, NVQ_F32 = 0, 1
STATUS_NAMES = {0: "NVQ_OK", 1: "NVQ_ERR_ARG", 2: "NVQ_ERR_SHAPE", 3: "NVQ_ERR_ALIGN", 4: "NVQ_ERR_CUDA",
                5: "NVQ_ERR_TIMEOUT"}


class NvqError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn} -> {STATUS_NAMES.get(status, status)}: {msg}")
        self.status = status


def _load():
    path = _build.build()
    lib = C.CDLL(path)
    for name, (args, res) in _SIGS.items():
        f = getattr(lib, name)
        f.argtypes = args
        f.restype = res
    return lib


LIB = _load()
LIB_PATH = _build.LIB


def _ptr(t):
    """Address of a buffer argument (None -> NULL).  Every buffer the library takes is device
    memory; a host tensor would reach a kernel as an invalid address, so it is refused here."""
    if t is None:
        return None
    if isinstance(t, torch.Tensor):
        if not t.is_cuda:
            raise ValueError(f"expected a CUDA tensor, got a tensor on {t.device}")
        return C.c_void_p(t.data_ptr())
    return C.c_void_p(t)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise NvqError(fn, status, LIB.nvq_last_error().decode())


# --------------------------------------------------------------------------- layout helpers
def sf_cols(ktot: int) -> int:
    return int(LIB.nvq_sf_cols(ktot))


def sf_bytes(rows: int, cols: int) -> int:
    return int(LIB.nvq_sf_bytes(rows, cols))


def sf_offset(row: int, col: int, cols: int) -> int:
    return int(LIB.nvq_sf_offset(row, col, cols))


def moe_capacity(tokens: int, topk: int, groups: int) -> int:
    return int(LIB.moe_capacity(tokens, topk, groups))


def moe_dispatch_workspace_size(tokens: int, topk: int, groups: int) -> int:
    return int(LIB.moe_dispatch_workspace_size(tokens, topk, groups))


def set_wait_limit(cycles: int):
    _check("nvq_set_wait_limit", LIB.nvq_set_wait_limit(cycles))


NVQ_TAIL_AUTO, NVQ_TAIL_GATHER, NVQ_TAIL_ROWS = 0, 1, 2


def set_tail_path(path: int):
    _check("nvq_set_tail_path", LIB.nvq_set_tail_path(path))


def device_status(stream=None):
    st, wh = C.c_int32(0), C.c_int32(0)
    _check("nvq_device_status", LIB.nvq_device_status(_stream(stream), C.byref(st), C.byref(wh)))
    return st.value, wh.value


def fp4_mma_rate(mmas_per_sm: int = 65536, with_cp: bool = False, stream=None) -> float:
    """Measured TFLOP/s of back-to-back NVFP4 MMAs on every SM (no memory traffic)."""
    v = C.c_float(0.0)
    _check("nvq_fp4_mma_rate", LIB.nvq_fp4_mma_rate(mmas_per_sm, int(bool(with_cp)), C.byref(v), _stream(stream)))
    return float(v.value)


def check_block_scale_division(result, stream=None):
    """result: CUDA uint32/int32 tensor of 2: [mismatch count, lowest mismatching bf16 pattern]."""
    _check("nvq_check_block_scale_division", LIB.nvq_check_block_scale_division(_ptr(result), _stream(stream)))


# --------------------------------------------------------------------------- the C ABI calls
def nvfp4_amax(x, tscale, grp_off=None, grp_rows=None, groups=1, rows=None, K=None, stream=None):
    rows = x.shape[0] if rows is None else rows
    K = x.shape[1] if K is None else K
    _check("nvfp4_amax", LIB.nvfp4_amax(_ptr(x), rows, K, x.stride(0), _ptr(grp_off), _ptr(grp_rows), groups,
                                        _ptr(tscale), _stream(stream)))


def nvfp4_quantize(x, codes, sf, sf_cols_, tscale, scores=None, grp_off=None, grp_rows=None, groups=1,
                   zero_pad=False, rows=None, K=None, amax_given=False, stream=None):
    rows = x.shape[0] if rows is None else rows
    K = x.shape[1] if K is None else K
    _check("nvfp4_quantize", LIB.nvfp4_quantize(
        _ptr(x), rows, K, x.stride(0), _ptr(grp_off), _ptr(grp_rows), groups, _ptr(codes), codes.stride(0),
        _ptr(sf), sf_cols_, int(bool(zero_pad)), _ptr(tscale), _ptr(scores), int(bool(amax_given)), _stream(stream)))


def rac_select_quantize(x, tscale, scores, k, codes, sf, sf_cols_, idx, grp_off=None, grp_rows=None, groups=1,
                        rows=None, K=None, stream=None):
    rows = x.shape[0] if rows is None else rows
    K = x.shape[1] if K is None else K
    _check("rac_select_quantize", LIB.rac_select_quantize(
        _ptr(x), rows, K, x.stride(0), _ptr(grp_off), _ptr(grp_rows), groups, _ptr(tscale), _ptr(scores), k,
        _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, _ptr(idx), _stream(stream)))


def weight_qdq(w, groups, N, K, codes, sf, sf_cols_, tscale, w_hat=None, w_hat_dtype=NVQ_BF16, stream=None):
    _check("weight_qdq", LIB.weight_qdq(
        _ptr(w), groups, N, K, w.stride(-2), _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, _ptr(tscale),
        _ptr(w_hat), w_hat_dtype, _stream(stream)))


def rac_select(scores, K, k, idx, groups=1, stream=None):
    _check("rac_select", LIB.rac_select(_ptr(scores), K, groups, k, _ptr(idx), _stream(stream)))


def rac_residual_tail(x, tscale, idx, k, codes, sf, sf_cols_, grp_off=None, grp_rows=None, groups=1, rows=None, K=None,
                      stream=None):
    rows = x.shape[0] if rows is None else rows
    K = x.shape[1] if K is None else K
    _check("rac_residual_tail", LIB.rac_residual_tail(
        _ptr(x), rows, K, x.stride(0), _ptr(grp_off), _ptr(grp_rows), groups, _ptr(tscale), _ptr(idx), k,
        _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, _stream(stream)))


def rac_reconstruct(codes, sf, sf_cols_, tscale, K, k, idx, out, rows=None, grp_off=None, grp_rows=None, groups=1,
                    stream=None):
    rows = codes.shape[0] if rows is None else rows
    _check("rac_reconstruct", LIB.rac_reconstruct(
        _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, _ptr(tscale), rows, K, k, _ptr(idx), _ptr(grp_off),
        _ptr(grp_rows), groups, _ptr(out), out.stride(0), _stream(stream)))


def w4a4_rac_grouped_gemm(a_codes, a_sf, a_sf_cols, a_tscale, b_codes, b_sf, b_sf_cols, b_tscale, N, K, k, idx,
                          out, groups=1, grp_off=None, grp_rows=None, rows=None, a_scale_per_group=False,
                          idx_per_group=False, epilogue=NVQ_EPI_STORE, row_w=None, out_tscale=None, stream=None):
    rows = a_codes.shape[0] if rows is None else rows
    _check("w4a4_rac_grouped_gemm", LIB.w4a4_rac_grouped_gemm(
        groups, _ptr(grp_off), _ptr(grp_rows), rows, _ptr(a_codes), a_codes.stride(0), _ptr(a_sf), a_sf_cols,
        _ptr(a_tscale), int(bool(a_scale_per_group)), _ptr(b_codes), b_codes.stride(0), _ptr(b_sf), b_sf_cols,
        _ptr(b_tscale), N, K, k, _ptr(idx), int(bool(idx_per_group)), epilogue, _ptr(row_w), _ptr(out),
        out.stride(0), _ptr(out_tscale), _stream(stream)))


def rac_weight_tail(groups, N, K, k, idx, b_codes, b_sf, b_sf_cols, b_tscale, idx_per_group=False, cm_codes=None,
                    cm_sf=None, stream=None):
    _check("rac_weight_tail", LIB.rac_weight_tail(
        groups, N, K, k, _ptr(idx), int(bool(idx_per_group)), _ptr(b_codes), b_codes.stride(0), _ptr(b_sf),
        b_sf_cols, _ptr(b_tscale), _ptr(cm_codes), _ptr(cm_sf), _stream(stream)))


def nvfp4_channel_major(groups, N, K, b_codes, b_sf, b_sf_cols, cm_codes, cm_sf, stream=None):
    _check("nvfp4_channel_major", LIB.nvfp4_channel_major(
        groups, N, K, _ptr(b_codes), b_codes.stride(0), _ptr(b_sf), b_sf_cols, _ptr(cm_codes), _ptr(cm_sf),
        _stream(stream)))


def moe_dispatch(topk_ids, topk_w, groups, grp_off, grp_rows, row_src, row_of, row_w, workspace, stream=None):
    T, topk = topk_ids.shape
    _check("moe_dispatch", LIB.moe_dispatch(
        _ptr(topk_ids), _ptr(topk_w), T, topk, groups, _ptr(grp_off), _ptr(grp_rows), _ptr(row_src), _ptr(row_of),
        _ptr(row_w), row_src.numel(), _ptr(workspace), workspace.numel(), _stream(stream)))


def moe_dispatch_static_scratch(topk_ids, topk_w, groups, grp_off, grp_rows, row_src, row_of, row_w, stream=None):
    """moe_dispatch with no workspace: the library's own 1 MiB device array holds the scratch.
    For callers that cannot allocate, or pass a workspace, where they dispatch. Calls that
    overlap on one device race on that array; the first call on a device does a one-time
    symbol lookup and should come before any stream capture."""
    T, topk = topk_ids.shape
    _check("moe_dispatch_static_scratch", LIB.moe_dispatch_static_scratch(
        _ptr(topk_ids), _ptr(topk_w), T, topk, groups, _ptr(grp_off), _ptr(grp_rows), _ptr(row_src), _ptr(row_of),
        _ptr(row_w), row_src.numel(), _stream(stream)))


def nvfp4_gather_rows(codes, sf, sf_cols_, src_rows, row_src, topk, ktot, out_codes, out_sf, col0=0, stream=None):
    _check("nvfp4_gather_rows", LIB.nvfp4_gather_rows(
        _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, src_rows, _ptr(row_src), topk, row_src.numel(), ktot, col0,
        _ptr(out_codes), out_codes.stride(0) if out_codes is not None else 0, _ptr(out_sf), _stream(stream)))


def fp8_sf_cols(K: int) -> int:
    return int(LIB.nvq_fp8_sf_cols(K))


def fp8_quantize(x, codes, sf, sf_cols_, tile_rows=1, rows=None, K=None, stream=None):
    rows = x.shape[0] if rows is None else rows
    K = x.shape[-1] if K is None else K
    _check("fp8_quantize", LIB.fp8_quantize(
        _ptr(x), rows, K, x.stride(-2), tile_rows, _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, _stream(stream)))


def fp8_blockscaled_grouped_gemm(a_codes, a_sf, a_sf_cols, b_codes, b_sf, b_sf_cols, N, K, out, groups=1, grp_off=None,
                                 grp_rows=None, rows=None, epilogue=NVQ_EPI_STORE, row_w=None, stream=None):
    rows = a_codes.shape[0] if rows is None else rows
    _check("fp8_blockscaled_grouped_gemm", LIB.fp8_blockscaled_grouped_gemm(
        groups, _ptr(grp_off), _ptr(grp_rows), rows, _ptr(a_codes), a_codes.stride(0), _ptr(a_sf), a_sf_cols,
        _ptr(b_codes), b_codes.stride(0), _ptr(b_sf), b_sf_cols, N, K, epilogue, _ptr(row_w), _ptr(out), out.stride(0),
        _stream(stream)))


def fp8_gather_rows(codes, sf, sf_cols_, src_rows, row_src, topk, K, out_codes, out_sf, stream=None):
    _check("fp8_gather_rows", LIB.fp8_gather_rows(
        _ptr(codes), codes.stride(0), _ptr(sf), sf_cols_, src_rows, _ptr(row_src), topk, row_src.numel(), K,
        _ptr(out_codes), out_codes.stride(0), _ptr(out_sf), _stream(stream)))


def moe_combine(y, row_of, tokens, topk, hidden, out, stream=None):
    _check("moe_combine", LIB.moe_combine(
        _ptr(y), y.stride(0), _ptr(row_of), tokens, topk, hidden, _ptr(out), out.stride(0), _stream(stream)))
