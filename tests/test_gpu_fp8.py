"""FP8 W8A8 block-scaled baseline on the GPU against the oracle: the quantizer bit for bit
(codes and UE8M0 tile scales in the blocked layout, 1 x 128 activation and 128 x 128 weight
tiles, ragged edges), the E4M3 conversion on every bf16 value, the row gather, and the
block-scaled grouped GEMM (bf16 out) within the GEMM tolerance of the fp64 product of the
dequantized operands, with the store, SwiGLU and routing-weight epilogues."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_testutil import GEMM_RTOL, bf16_bits, bf16_tensor, gemm_error, unswizzle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    return _lib


def _quant(L, x_bits, tile_rows):
    R, K = x_bits.shape
    ld = (K + 15) // 16 * 16
    sfc = L.fp8_sf_cols(K)
    codes = torch.full((R, ld), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((L.sf_bytes(R, sfc),), 0xCD, dtype=torch.uint8, device="cuda")
    L.fp8_quantize(bf16_tensor(x_bits), codes, sf, sfc, tile_rows=tile_rows)
    torch.cuda.synchronize()
    return codes, sf, sfc


def _expected_sf(st, rows, K, tile_rows):
    """Logical [rows][roundup(K/32, 4)] scale bytes: the tile byte on its 4 columns (and
    tile_rows rows), zero on the columns of the last word beyond K / 32."""
    ncols = (K // 32 + 3) // 4 * 4
    out = np.zeros((rows, ncols), np.uint8)
    for r in range(rows):
        for j in range(K // 32):
            out[r, j] = st[r // tile_rows, j // 4]
    return out


@pytest.mark.parametrize("M,K", [(64, 256), (130, 768), (3, 4096), (257, 2144), (1, 32)])
def test_fp8_quantize_activations(L, M, K):
    x, _ = wl.activations(M, K, seed=M + K, dist="student_t3", scale=0.5, n_outliers=max(1, K // 100), outlier_gain=20.0)
    codes, sf, sfc = _quant(L, x, 1)
    oc, st = oracle.fp8_quantize(x, 1)
    assert np.array_equal(codes.cpu().numpy()[:, :K], oc)
    assert np.array_equal(unswizzle(sf, M, (K // 32 + 3) // 4 * 4, sfc), _expected_sf(st, M, K, 1))


@pytest.mark.parametrize("R,K", [(256, 384), (384, 800), (128, 2048), (200, 96)])
def test_fp8_quantize_weights(L, R, K):
    w = wl.weights((R, K), 0.02, seed=R + K)
    wf = wl.bf16_bits_to_f32(w).astype(np.float64)
    wf[R // 3, K // 2] = 3.0  # one outlier: only its tile's scale moves
    w = wl.to_bf16_bits(wf)
    codes, sf, sfc = _quant(L, w, 128)
    oc, st = oracle.fp8_quantize(w, 128)
    assert np.array_equal(codes.cpu().numpy()[:, :K], oc)
    assert np.array_equal(unswizzle(sf, R, (K // 32 + 3) // 4 * 4, sfc), _expected_sf(st, R, K, 128))


def test_fp8_encode_every_bf16_value(L):
    """Tiles whose first element is 448 have e = 0, so every other element's code is the plain
    E4M3 conversion: checked against the oracle for every finite bf16 value up to 448."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        v = wl.bf16_bits_to_f32(bits).astype(np.float64)
    vals = bits[np.isfinite(v) & (np.abs(v) <= 448.0)]
    per = 127
    n = (vals.size + per - 1) // per
    x = np.zeros((n, 128), np.uint16)
    x[:, 0] = wl.to_bf16_bits(np.array([448.0]))[0]
    flat = np.zeros(n * per, np.uint16)
    flat[:vals.size] = vals
    x[:, 1:] = flat.reshape(n, per)
    codes, _, _ = _quant(L, x, 1)
    got = codes.cpu().numpy()[:, 1:].ravel()[:vals.size]
    ref = np.array([oracle.lib().oracle_fp8_encode(float(t)) for t in wl.bf16_bits_to_f32(vals).astype(np.float64)], np.uint8)
    assert np.array_equal(got, ref)


def _gemm_case(L, counts, N, K, epilogue, seed, dense=False):
    G = len(counts)
    off = [0]
    for c in counts:
        off.append(off[-1] + (c if dense else (c + 127) // 128 * 128))
    rows = max(off[-1], 1)
    sfc = L.fp8_sf_cols(K)
    ld = (K + 15) // 16 * 16
    a_codes = torch.zeros(rows, ld, dtype=torch.uint8, device="cuda")
    a_sf = torch.zeros(L.sf_bytes(rows, sfc), dtype=torch.uint8, device="cuda")
    x = np.zeros((rows, K), np.uint16)
    for g, c in enumerate(counts):
        if c:
            xg, _ = wl.activations(c, K, seed=seed * 10 + g, n_outliers=max(1, K // 64), outlier_gain=12.0)
            x[off[g]:off[g] + c] = xg
    L.fp8_quantize(bf16_tensor(x), a_codes, a_sf, sfc, tile_rows=1)
    w = wl.weights((G * N, K), 0.02, seed=seed + 77)
    b_codes = torch.zeros(G * N, ld, dtype=torch.uint8, device="cuda")
    b_sf = torch.zeros(L.sf_bytes(G * N, sfc), dtype=torch.uint8, device="cuda")
    L.fp8_quantize(bf16_tensor(w), b_codes, b_sf, sfc, tile_rows=128)
    row_w = torch.from_numpy(np.random.default_rng(seed).uniform(0.1, 1.0, rows).astype(np.float32)).cuda()
    width = N // 2 if epilogue == L.NVQ_EPI_SWIGLU else N
    out = torch.zeros(rows, width, dtype=torch.bfloat16, device="cuda")
    go = torch.tensor(off, dtype=torch.int64, device="cuda")
    gr = torch.tensor(counts, dtype=torch.int64, device="cuda")
    L.fp8_blockscaled_grouped_gemm(a_codes, a_sf, sfc, b_codes, b_sf, sfc, N, K, out, groups=G,
                                   grp_off=go if G > 1 else None, grp_rows=gr if G > 1 else None, rows=rows,
                                   epilogue=epilogue, row_w=row_w if epilogue == L.NVQ_EPI_ROW_SCALE else None)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    y = wl.bf16_bits_to_f32(bf16_bits(out))
    worst = 0.0
    rw = row_w.cpu().numpy().astype(np.float64)
    for g, c in enumerate(counts):
        if not c:
            continue
        ac, ast = oracle.fp8_quantize(x[off[g]:off[g] + c], 1)
        bc, bst = oracle.fp8_quantize(w[g * N:(g + 1) * N], 128)
        ref = oracle.fp8_gemm(ac, ast, bc, bst)
        if epilogue == L.NVQ_EPI_SWIGLU:
            ref = oracle.swiglu(ref[:, :N // 2], ref[:, N // 2:]).reshape(c, N // 2)
        elif epilogue == L.NVQ_EPI_ROW_SCALE:
            ref = ref * rw[off[g]:off[g] + c, None]
        worst = max(worst, gemm_error(y[off[g]:off[g] + c], ref))
    assert worst <= GEMM_RTOL, worst
    return worst


@pytest.mark.parametrize("M,N,K", [(128, 256, 256), (300, 512, 768), (1, 256, 128), (77, 768, 2080), (256, 256, 4096)])
def test_fp8_gemm_dense(L, M, N, K):
    _gemm_case(L, [M], N, K, 0, seed=M + K, dense=True)


@pytest.mark.parametrize("epilogue", [1, 2])
def test_fp8_gemm_grouped_epilogues(L, epilogue):
    _gemm_case(L, [5, 0, 300, 129], 512, 256, epilogue, seed=60 + epilogue)


def test_fp8_gather_rows(L):
    T, K, topk, E = 200, 768, 2, 4
    x, _ = wl.activations(T, K, seed=90, n_outliers=4, outlier_gain=10.0)
    codes, sf, sfc = _quant(L, x, 1)
    ids, _ = wl.routing_uniform(T, E, topk, seed=91)
    cap = L.moe_capacity(T, topk, E)
    o_off, o_src = oracle.moe_dispatch(ids, E)
    row_src = np.full(cap, -1, np.int32)
    off = 0
    for g in range(E):
        c = o_off[g + 1] - o_off[g]
        row_src[off:off + c] = o_src[o_off[g]:o_off[g + 1]]
        off += (c + 127) // 128 * 128
    rs = torch.from_numpy(row_src).cuda()
    out_codes = torch.full((cap, codes.shape[1]), 0x55, dtype=torch.uint8, device="cuda")
    out_sf = torch.full((L.sf_bytes(cap, sfc),), 0x55, dtype=torch.uint8, device="cuda")
    L.fp8_gather_rows(codes, sf, sfc, T, rs, topk, K, out_codes, out_sf)
    torch.cuda.synchronize()
    src_c = codes.cpu().numpy()[:, :K]
    src_s = unswizzle(sf, T, sfc, sfc)
    got_c = out_codes.cpu().numpy()[:, :K]
    got_s = unswizzle(out_sf, cap, sfc, sfc)
    for i in range(cap):
        if row_src[i] >= 0:
            t = row_src[i] // topk
            assert np.array_equal(got_c[i], src_c[t]) and np.array_equal(got_s[i], src_s[t])
        else:
            assert not got_c[i].any() and not got_s[i].any()


def test_fp8_moe_layer_stages(L):
    """Fp8MoELayer on a small Zipf-routed batch, stage by stage against the oracle: token codes
    and scales bit for bit, gate/up + SwiGLU and down + routing weight within the GEMM
    tolerance (each from the GPU's own previous stage), h codes bit for bit, combine exact."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Fp8MoELayer
    T, H, E, topk, I = 300, 256, 8, 2, 128
    cfg = wl.MoELayer("t", T=T, H=H, E=E, topk=topk, I=I, k=0, seed=25, routing="zipf", n_outliers=3)
    x_bits, ids, tw, _ = cfg.make_tokens()
    w13_bits, w2_bits = cfg.make_weights()
    w13 = bf16_tensor(w13_bits.reshape(E * 2 * I, H)).view(E, 2 * I, H)
    w2 = bf16_tensor(w2_bits.reshape(E * H, I)).view(E, H, I)
    layer = Fp8MoELayer(w13, w2, topk, T)
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    layer.forward(bf16_tensor(x_bits), torch.from_numpy(ids).cuda(), torch.from_numpy(tw).cuda(), out)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    tc, tst = oracle.fp8_quantize(x_bits, 1)
    assert np.array_equal(layer.a_tok.codes.cpu().numpy()[:, :H], tc)
    assert np.array_equal(unswizzle(layer.a_tok.sf, T, layer.a_tok.sf_cols, layer.a_tok.sf_cols),
                          _expected_sf(tst, T, H, 1))
    grp_off = layer.grp_off.cpu().numpy()
    grp_rows = layer.grp_rows.cpu().numpy()
    row_src = layer.row_src.cpu().numpy()
    row_w = layer.row_w.cpu().numpy().astype(np.float64)
    h_gpu = bf16_bits(layer.h)
    y_gpu = bf16_bits(layer.y)
    worst_h = worst_y = 0.0
    for g in range(E):
        c = int(grp_rows[g])
        if not c:
            continue
        rows = np.arange(grp_off[g], grp_off[g] + c)
        toks = row_src[rows] // topk
        w13c, w13s = oracle.fp8_quantize(w13_bits[g], 128)
        ref = oracle.fp8_gemm(tc[toks], tst[toks], w13c, w13s)
        href = oracle.swiglu(ref[:, :I], ref[:, I:]).reshape(c, I)
        worst_h = max(worst_h, gemm_error(wl.bf16_bits_to_f32(h_gpu[rows]), href))
        hc, hst = oracle.fp8_quantize(h_gpu[rows], 1)
        assert np.array_equal(layer.a2.codes.cpu().numpy()[rows][:, :I], hc)
        w2c, w2s = oracle.fp8_quantize(w2_bits[g], 128)
        yref = oracle.fp8_gemm(hc, hst, w2c, w2s) * row_w[rows][:, None]
        worst_y = max(worst_y, gemm_error(wl.bf16_bits_to_f32(y_gpu[rows]), yref))
    assert worst_h <= GEMM_RTOL and worst_y <= GEMM_RTOL, (worst_h, worst_y)
    pos = layer.row_of.cpu().numpy()
    assert np.array_equal(bf16_bits(out), oracle.moe_combine(y_gpu, pos, topk))
