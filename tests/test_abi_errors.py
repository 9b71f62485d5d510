"""Argument errors of the C ABI, on the CPU: every entry below validates its arguments on the
host before any CUDA call, so bad shapes, alignments, enumerators and null pointers come back as
the status codes include/nvfp4rac.h documents (with nvq_last_error naming the entry) without a
GPU.  The pointers are placeholders the entries never dereference."""
import ctypes as C

import pytest

from nvfp4_w4a4_quantized_quantize_gb300 import _lib as Lmod

LIB = Lmod.LIB
OK, ARG, SHAPE, ALIGN = 0, 1, 2, 3
P = 0x100000        # a 256-byte-aligned placeholder address
ODD = 0x100001      # a misaligned one


def _err():
    return LIB.nvq_last_error().decode()


def _fp8_quantize(x=P, rows=64, K=256, ldx=256, tile_rows=1, codes=P, ld_codes=256, sf=P, sf_cols=8):
    return LIB.fp8_quantize(x, rows, K, ldx, tile_rows, codes, ld_codes, sf, sf_cols, None)


@pytest.mark.parametrize("kw,status", [
    (dict(K=48), SHAPE), (dict(K=16), SHAPE), (dict(tile_rows=64), ARG), (dict(x=0), ARG),
    (dict(codes=ODD), ALIGN), (dict(ldx=100), ALIGN), (dict(sf_cols=4), SHAPE), (dict(rows=0), SHAPE),
])
def test_fp8_quantize_argument_errors(kw, status):
    assert _fp8_quantize(**kw) == status
    assert _err().startswith("fp8_quantize")


def _fp8_gemm(groups=1, grp_off=0, rows=128, a=P, lda=256, a_sf=P, a_sfc=8, b=P, ldb=256, b_sf=P, b_sfc=8, N=256,
              K=256, epi=0, row_w=0, out=P, ldo=256):
    return LIB.fp8_blockscaled_grouped_gemm(groups, grp_off, 0, rows, a, lda, a_sf, a_sfc, b, ldb, b_sf, b_sfc, N, K,
                                            epi, row_w, out, ldo, None)


@pytest.mark.parametrize("kw,status", [
    (dict(N=100), SHAPE), (dict(epi=9), ARG), (dict(epi=2), ARG), (dict(K=48), SHAPE), (dict(lda=8), ALIGN),
    (dict(groups=2), SHAPE), (dict(a_sfc=4, K=512, lda=512, ldb=512, b_sfc=16), SHAPE), (dict(out=ODD), ALIGN), (dict(b=0), ARG),
])
def test_fp8_gemm_argument_errors(kw, status):
    assert _fp8_gemm(**kw) == status
    assert _err().startswith("fp8_blockscaled_grouped_gemm")


@pytest.mark.parametrize("kw,status", [(dict(capacity=100), SHAPE), (dict(K=20), SHAPE), (dict(row_src=0), ARG),
                                       (dict(ld_codes=8), ALIGN)])
def test_fp8_gather_rows_argument_errors(kw, status):
    a = dict(codes=P, ld_codes=256, sf=P, sf_cols=8, src_rows=10, row_src=P, topk=2, capacity=128, K=256,
             out_codes=P, ld_out=256, out_sf=P)
    a.update(kw)
    assert LIB.fp8_gather_rows(a["codes"], a["ld_codes"], a["sf"], a["sf_cols"], a["src_rows"], a["row_src"], a["topk"],
                               a["capacity"], a["K"], a["out_codes"], a["ld_out"], a["out_sf"], None) == status
    assert _err().startswith("fp8_gather_rows")


@pytest.mark.parametrize("kw,status", [(dict(k=24), SHAPE), (dict(k=512), SHAPE), (dict(out=ODD), ALIGN),
                                       (dict(ldo=128), SHAPE), (dict(idx=0), ARG), (dict(groups=3), SHAPE),
                                       (dict(K=40), SHAPE)])
def test_rac_reconstruct_argument_errors(kw, status):
    a = dict(codes=P, ld_codes=256, sf=P, sf_cols=24, ts=P, rows=64, K=256, k=32, idx=P, grp_off=0, grp_rows=0,
             groups=1, out=P, ldo=256)
    a.update(kw)
    assert LIB.rac_reconstruct(a["codes"], a["ld_codes"], a["sf"], a["sf_cols"], a["ts"], a["rows"], a["K"], a["k"],
                               a["idx"], a["grp_off"], a["grp_rows"], a["groups"], a["out"], a["ldo"], None) == status
    assert _err().startswith("rac_reconstruct")


def test_tail_path_setting():
    assert LIB.nvq_set_tail_path(7) == ARG and "nvq_set_tail_path" in _err()
    for p in (Lmod.NVQ_TAIL_ROWS, Lmod.NVQ_TAIL_GATHER, Lmod.NVQ_TAIL_AUTO):
        assert LIB.nvq_set_tail_path(p) == OK


def test_fp8_layout_helper():
    assert [Lmod.fp8_sf_cols(K) for K in (32, 128, 160, 768, 2048, 2080)] == [4, 4, 8, 24, 64, 68]


def test_binding_refuses_host_tensors():
    """A host tensor handed to the binding is refused before the library sees its address."""
    import torch
    x = torch.zeros(4, 32, dtype=torch.bfloat16)
    codes = torch.zeros(4, 32, dtype=torch.uint8)
    sf = torch.zeros(512, dtype=torch.uint8)
    with pytest.raises(ValueError, match="CUDA tensor"):
        Lmod.fp8_quantize(x, codes, sf, 4)


@pytest.mark.parametrize("mmas,out", [(8, True), (1 << 21, True), (1024, False)])
def test_mma_rate_probe_argument_errors(mmas, out):
    """nvq_fp4_mma_rate refuses a loop shorter than 16 or longer than 2^20 MMAs per SM and a NULL
    result pointer before it touches the GPU."""
    v = C.c_float(0.0)
    assert LIB.nvq_fp4_mma_rate(mmas, 0, C.byref(v) if out else None, None) == ARG
    assert _err().startswith("nvq_fp4_mma_rate")
