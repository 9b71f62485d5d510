"""CPU oracle for the NVFP4 W4A4 + Residual Activation Compensation path (test infrastructure).

Only the test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may
import this package.  It wraps ``nvfp4_oracle.c`` (plain scalar C, compiled here with gcc and
``-ffp-contract=off``) and shares no code with the CUDA library.

Everything follows "QUADS: Stabilizing NVFP4 Reinforcement Learning for MoE via
QUantization-error Alignment across Dual Sides" (arXiv 2607.15810): §2.2 "FP4"/"FP8" for the
formats, Eq. (7)/(9)/(12) for the QDQ operators, Eq. (20)-(24) for the residual compensation.
The readings of the points the paper leaves open are listed in the header of the C file.
Parity unpinned (conventions no value printed in the paper can confirm): the per-tensor scale
formula, the block-scale operation order, the weight-tail reading and the per-expert scope of
the down-projection's tensor scale.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libnvfp4_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (portable C11, no FMA contraction, no target flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", _SRC, "-o", tmp, "-lm", "-lpthread"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _TScale(C.Structure):
    _fields_ = [("amax", C.c_float), ("s_enc", C.c_float), ("s_dec", C.c_float),
                ("shift_e", C.c_int32)]


@dataclass
class TensorScale:
    """Per-tensor FP32 scale (QUADS §2.2 "FP4", second scaling level)."""
    amax: float
    s_enc: float
    s_dec: float
    shift_e: int

    def _c(self) -> _TScale:
        return _TScale(self.amax, self.s_enc, self.s_dec, self.shift_e)


def lib():
    global _lib
    if _lib is None:
        _lib = C.CDLL(build())
        P, I64, I32 = C.c_void_p, C.c_int64, C.c_int32
        sig = {
            "oracle_bf16_round": ([C.c_float], C.c_uint16),
            "oracle_bf16_value": ([C.c_uint16], C.c_float),
            "oracle_e2m1_value": ([C.c_uint8], C.c_double),
            "oracle_e2m1_encode": ([C.c_float], C.c_uint8),
            "oracle_e4m3_value": ([C.c_uint8], C.c_double),
            "oracle_e4m3_encode": ([C.c_float], C.c_uint8),
            "oracle_tensor_scale": ([P, I64, I64, I64, P], None),
            "oracle_tensor_scale_from_amax": ([C.c_float, P], None),
            "oracle_quantize": ([P, I64, I64, I64, P, P, I64, P, I64], None),
            "oracle_dequantize": ([P, I64, P, I64, I64, I64, C.c_float, P, I64], None),
            "oracle_residual": ([P, I64, I64, I64, P, P, I64], None),
            "oracle_scores": ([P, I64, I64, I64, P, P], None),
            "oracle_topk": ([P, I64, I32, P], None),
            "oracle_rac_tail": ([P, I64, I64, I64, P, P, I32, P, I64, P, I64], None),
            "oracle_weight_tail": ([P, I64, P, I64, I64, P, P, I32, P, I64, P, I64], None),
            "oracle_gemm_pairs": ([P, I64, P, I64, P, I64, P, I64, I64, C.c_double, C.c_double,
                                   P, P, I64, P], None),
            "oracle_gemm_pairs_fp64": ([P, I64, P, I64, P, I64, P, I64, I64, C.c_double,
                                        C.c_double, P, P, I64, P], None),
            "oracle_moe_dispatch": ([P, I64, I32, I32, P, P], None),
            "oracle_swiglu": ([C.c_double, C.c_double], C.c_double),
            "oracle_moe_combine": ([P, I64, P, I64, I32, I64, P, I64], None),
            "oracle_e2m1_encode_array": ([P, I64, P], None),
            "oracle_e4m3_encode_array": ([P, I64, P], None),
            "oracle_bf16_round_array": ([P, I64, P], None),
            "oracle_quantize_block16": ([P, C.c_float, P, P], None),
            "oracle_fp8_scale_exponent": ([C.c_double], C.c_int32),
            "oracle_fp8_encode": ([C.c_double], C.c_uint8),
            "oracle_fp8_quantize": ([P, I64, I64, I64, I32, P, I64, P, I64], None),
            "oracle_fp8_dequantize": ([P, I64, P, I64, I64, I64, I32, P, I64], None),
            "oracle_set_threads": ([C.c_int], None),
            "oracle_hardware_threads": ([], C.c_int),
        }
        for name, (args, res) in sig.items():
            f = getattr(_lib, name)
            f.argtypes = args
            f.restype = res
    return _lib


def set_threads(n: int) -> None:
    """Host threads the GEMM's output pairs are spread over (the result does not depend on it)."""
    lib().oracle_set_threads(int(n))


def hardware_threads() -> int:
    return int(lib().oracle_hardware_threads())


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(C.c_void_p)


def _bf16(x: np.ndarray) -> np.ndarray:
    assert x.dtype == np.uint16, "bf16 inputs are passed as their uint16 bit patterns"
    return np.ascontiguousarray(x)


# ---------------------------------------------------------------- element formats
def e2m1_value(code: int) -> float:
    return lib().oracle_e2m1_value(code)


def e4m3_value(b: int) -> float:
    return lib().oracle_e4m3_value(b)


def e2m1_encode(v: np.ndarray) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().oracle_e2m1_encode_array(_p(v), v.size, _p(out))
    return out


def e4m3_encode(t: np.ndarray) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float32)
    out = np.empty(t.shape, np.uint8)
    lib().oracle_e4m3_encode_array(_p(t), t.size, _p(out))
    return out


def bf16_round(f: np.ndarray) -> np.ndarray:
    f = np.ascontiguousarray(f, dtype=np.float32)
    out = np.empty(f.shape, np.uint16)
    lib().oracle_bf16_round_array(_p(f), f.size, _p(out))
    return out


def quantize_block16(v: np.ndarray, s_enc: float):
    v = np.ascontiguousarray(v, dtype=np.float32)
    assert v.size == 16
    codes = np.empty(16, np.uint8)
    sb = np.empty(1, np.uint8)
    lib().oracle_quantize_block16(_p(v), C.c_float(s_enc), _p(codes), _p(sb))
    return codes, int(sb[0])


# ---------------------------------------------------------------- quantizer (Q_A / Q_W)
def tensor_scale(x: np.ndarray) -> TensorScale:
    x = _bf16(x)
    ts = _TScale()
    lib().oracle_tensor_scale(_p(x), x.shape[0], x.shape[1], x.shape[1], C.byref(ts))
    return TensorScale(ts.amax, ts.s_enc, ts.s_dec, ts.shift_e)


def tensor_scale_from_amax(amax: float) -> TensorScale:
    ts = _TScale()
    lib().oracle_tensor_scale_from_amax(C.c_float(amax), C.byref(ts))
    return TensorScale(ts.amax, ts.s_enc, ts.s_dec, ts.shift_e)


def quantize(x: np.ndarray, ts: TensorScale):
    """NVFP4 codes [R, C/2] (element 2i in the low nibble) and E4M3 scales [R, C/16]."""
    x = _bf16(x)
    R, Cc = x.shape
    assert Cc % 16 == 0
    codes = np.zeros((R, Cc // 2), np.uint8)
    scales = np.zeros((R, Cc // 16), np.uint8)
    t = ts._c()
    lib().oracle_quantize(_p(x), R, Cc, Cc, C.byref(t), _p(codes), Cc // 2, _p(scales), Cc // 16)
    return codes, scales


def dequantize(codes: np.ndarray, scales: np.ndarray, s_dec: float) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    R, half = codes.shape
    out = np.empty((R, half * 2), np.float32)
    lib().oracle_dequantize(_p(codes), half, _p(scales), scales.shape[1], R, half * 2,
                            C.c_float(s_dec), _p(out), half * 2)
    return out


def residual(x: np.ndarray, ts: TensorScale) -> np.ndarray:
    x = _bf16(x)
    R, Cc = x.shape
    r = np.empty((R, Cc), np.float32)
    t = ts._c()
    lib().oracle_residual(_p(x), R, Cc, Cc, C.byref(t), _p(r), Cc)
    return r


def scores(x: np.ndarray, ts: TensorScale) -> np.ndarray:
    x = _bf16(x)
    R, Cc = x.shape
    s = np.zeros(Cc, np.uint64)
    t = ts._c()
    lib().oracle_scores(_p(x), R, Cc, Cc, C.byref(t), _p(s))
    return s


def topk(s: np.ndarray, k: int) -> np.ndarray:
    s = np.ascontiguousarray(s, dtype=np.uint64)
    idx = np.zeros(k, np.int32)
    lib().oracle_topk(_p(s), s.size, k, _p(idx))
    return idx


def rac_tail(x: np.ndarray, ts: TensorScale, idx: np.ndarray):
    x = _bf16(x)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k = idx.size
    R, Cc = x.shape
    tc = np.zeros((R, k // 2), np.uint8)
    tsc = np.zeros((R, k // 16), np.uint8)
    t = ts._c()
    lib().oracle_rac_tail(_p(x), R, Cc, Cc, C.byref(t), _p(idx), k, _p(tc), k // 2, _p(tsc), k // 16)
    return tc, tsc


def weight_tail(wcodes: np.ndarray, wscales: np.ndarray, wts: TensorScale, idx: np.ndarray):
    wcodes = np.ascontiguousarray(wcodes)
    wscales = np.ascontiguousarray(wscales)
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    k = idx.size
    N = wcodes.shape[0]
    tc = np.zeros((N, k // 2), np.uint8)
    tsc = np.zeros((N, k // 16), np.uint8)
    t = wts._c()
    lib().oracle_weight_tail(_p(wcodes), wcodes.shape[1], _p(wscales), wscales.shape[1], N,
                             C.byref(t), _p(idx), k, _p(tc), k // 2, _p(tsc), k // 16)
    return tc, tsc


def _gemm(fn, a_codes, a_scales, b_codes, b_scales, s_dec_a, s_dec_b, mi, ni):
    a_codes, a_scales = np.ascontiguousarray(a_codes), np.ascontiguousarray(a_scales)
    b_codes, b_scales = np.ascontiguousarray(b_codes), np.ascontiguousarray(b_scales)
    mi = np.ascontiguousarray(mi, dtype=np.int64)
    ni = np.ascontiguousarray(ni, dtype=np.int64)
    ktot = a_codes.shape[1] * 2
    assert b_codes.shape[1] * 2 == ktot
    y = np.empty(mi.size, np.float64)
    fn(_p(a_codes), a_codes.shape[1], _p(a_scales), a_scales.shape[1], _p(b_codes),
       b_codes.shape[1], _p(b_scales), b_scales.shape[1], ktot, float(s_dec_a), float(s_dec_b),
       _p(mi), _p(ni), mi.size, _p(y))
    return y


def gemm_pairs(a_codes, a_scales, b_codes, b_scales, s_dec_a, s_dec_b, mi, ni) -> np.ndarray:
    """Exact block-scaled FP4 product at the (mi[p], ni[p]) output positions."""
    return _gemm(lib().oracle_gemm_pairs, a_codes, a_scales, b_codes, b_scales, s_dec_a, s_dec_b, mi, ni)


def gemm_pairs_fp64(a_codes, a_scales, b_codes, b_scales, s_dec_a, s_dec_b, mi, ni) -> np.ndarray:
    return _gemm(lib().oracle_gemm_pairs_fp64, a_codes, a_scales, b_codes, b_scales, s_dec_a,
                 s_dec_b, mi, ni)


def gemm(a_codes, a_scales, b_codes, b_scales, s_dec_a, s_dec_b) -> np.ndarray:
    M, N = a_codes.shape[0], b_codes.shape[0]
    mi, ni = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return gemm_pairs(a_codes, a_scales, b_codes, b_scales, s_dec_a, s_dec_b,
                      mi.ravel(), ni.ravel()).reshape(M, N)


# ---------------------------------------------------------------- MoE plumbing
def moe_dispatch(topk_ids: np.ndarray, groups: int):
    ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    T, topk = ids.shape
    grp_off = np.zeros(groups + 1, np.int64)
    row_src = np.zeros(T * topk, np.int32)
    lib().oracle_moe_dispatch(_p(ids), T, topk, groups, _p(grp_off), _p(row_src))
    return grp_off, row_src


def swiglu(g: np.ndarray, u: np.ndarray) -> np.ndarray:
    f = lib().oracle_swiglu
    g = np.asarray(g, np.float64).ravel()
    u = np.asarray(u, np.float64).ravel()
    return np.array([f(float(a), float(b)) for a, b in zip(g, u)], np.float64)


def moe_combine(y: np.ndarray, pos: np.ndarray, topk: int) -> np.ndarray:
    y = _bf16(y)
    pos = np.ascontiguousarray(pos, dtype=np.int64)
    T = pos.size // topk
    H = y.shape[1]
    out = np.zeros((T, H), np.uint16)
    lib().oracle_moe_combine(_p(y), H, _p(pos), T, topk, H, _p(out), H)
    return out


# ---------------------------------------------------------------- composed dense RAC linear
@dataclass
class RacQuant:
    ts: TensorScale
    codes: np.ndarray      # [M, K/2]
    scales: np.ndarray     # [M, K/16]
    scores: np.ndarray     # [K] uint64
    idx: np.ndarray        # [k] int32 ascending
    tail_codes: np.ndarray   # [M, k/2]
    tail_scales: np.ndarray  # [M, k/16]


def rac_reconstruct(q: RacQuant) -> np.ndarray:
    """The compensated activation of QUADS Eq. (21), X-tilde = DQ(Q(X)) + DQ(Q(R)) on the selected
    channels and DQ(Q(X)) elsewhere, as binary32: each dequantized value is fl(V * fl(sb * S_dec))
    (the `dequantize` above) and the two are summed with one binary32 addition (numpy float32
    arithmetic rounds to nearest-even)."""
    out = dequantize(q.codes, q.scales, q.ts.s_dec)
    if q.idx.size:
        tail = dequantize(q.tail_codes, q.tail_scales, q.ts.s_dec)
        out[:, q.idx] = out[:, q.idx] + tail
    return out


def rac_quantize(x: np.ndarray, k: int) -> RacQuant:
    """Steps of QUADS §3.3 in the paper's order: Q_A(X), residual, score, TopK, second pass."""
    ts = tensor_scale(x)
    codes, scales = quantize(x, ts)
    s = scores(x, ts)
    idx = topk(s, k) if k > 0 else np.zeros(0, np.int32)
    if k > 0:
        tc, tsc = rac_tail(x, ts, idx)
    else:
        tc = np.zeros((x.shape[0], 0), np.uint8)
        tsc = np.zeros((x.shape[0], 0), np.uint8)
    return RacQuant(ts, codes, scales, s, idx, tc, tsc)


# ---------------------------------------------------------------- FP8 W8A8 comparison baseline
# QUADS §2.2 "FP8" (E4M3, a scale per tile of values) and §4.4.2 (FP8 W8A8 rollout as the
# production baseline).  Tiles and scale encoding: readings R16-R18 of nvfp4_oracle.c.
def fp8_scale_exponent(amax: float) -> int:
    return int(lib().oracle_fp8_scale_exponent(float(amax)))


def fp8_quantize(x: np.ndarray, tile_rows: int):
    """bf16 bits [R, C] -> E4M3 codes [R, C] and UE8M0 tile bytes [ceil(R/tile_rows), ceil(C/128)]."""
    x = _bf16(x)
    R, Cc = x.shape
    codes = np.zeros((R, Cc), np.uint8)
    st = np.zeros(((R + tile_rows - 1) // tile_rows, (Cc + 127) // 128), np.uint8)
    lib().oracle_fp8_quantize(_p(x), R, Cc, Cc, tile_rows, _p(codes), Cc, _p(st), st.shape[1])
    return codes, st


def fp8_dequantize(codes: np.ndarray, scales: np.ndarray, tile_rows: int) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    R, Cc = codes.shape
    out = np.zeros((R, Cc), np.float64)
    lib().oracle_fp8_dequantize(_p(codes), Cc, _p(scales), scales.shape[1], R, Cc, tile_rows, _p(out), Cc)
    return out


def fp8_gemm(a_codes, a_scales, b_codes, b_scales) -> np.ndarray:
    """Y = DQ(A) DQ(B)^T in fp64 (A: 1 x 128 tiles, B: 128 x 128 tiles); the products of
    dequantized values are exact and the matmul accumulates in fp64."""
    return fp8_dequantize(a_codes, a_scales, 1) @ fp8_dequantize(b_codes, b_scales, 128).T
