"""GPU parity of the quantizer, the channel scores, the RAC selection and tails, and the
trainer-side weight QDQ against the CPU oracle: bit-exact codes, scales, scores and indices."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import bf16_tensor, tscale_fields, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 31)
    return _lib


@pytest.fixture
def tail_path(L, request):
    """Forces one schedule of the tail columns (nvq_set_tail_path) for the test, then restores auto."""
    L.set_tail_path(request.param)
    yield request.param
    L.set_tail_path(L.NVQ_TAIL_AUTO)


PATHS = pytest.mark.parametrize("tail_path", [1, 2], indirect=True, ids=["gather", "rows"])


def _gpu_quant(L, x_bits, k=0, groups=1, grp_off=None, grp_rows=None, ktail=None):
    M, K = x_bits.shape
    x = bf16_tensor(x_bits)
    ktot = K + (ktail if ktail is not None else k)
    ld = max(16, (ktot // 2 + 15) // 16 * 16)
    sf_cols = L.sf_cols(ktot)
    codes = torch.full((M, ld), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((L.sf_bytes(M, sf_cols),), 0xCD, dtype=torch.uint8, device="cuda")
    ts = torch.zeros(groups, 4, dtype=torch.float32, device="cuda")
    scores = torch.zeros(groups, K, dtype=torch.int64, device="cuda")
    go = torch.tensor(grp_off, dtype=torch.int64, device="cuda") if grp_off is not None else None
    gr = torch.tensor(grp_rows, dtype=torch.int64, device="cuda") if grp_rows is not None else None
    L.nvfp4_quantize(x, codes, sf, sf_cols, ts, scores=scores, grp_off=go, grp_rows=gr, groups=groups,
                     zero_pad=(k == 0))
    idx = torch.zeros(groups, max(k, 1), dtype=torch.int32, device="cuda")
    if k:
        L.rac_select_quantize(x, ts, scores, k, codes, sf, sf_cols, idx, grp_off=go, grp_rows=gr, groups=groups)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    return dict(codes=codes.cpu().numpy(), sf=sf, sf_cols=sf_cols, ts=ts, scores=scores.cpu().numpy().view(np.uint64),
                idx=idx.cpu().numpy(), codes_d=codes, idx_d=idx, go=go, gr=gr)


def _check_rows(L, x_bits, g, rows, k, K, ref_k=None):
    """Compare rows [rows] of the GPU result g against the oracle applied to those rows."""
    xs = x_bits[rows]
    ts = oracle.tensor_scale(xs)
    oc, os_ = oracle.quantize(xs, ts)
    assert np.array_equal(g["codes"][rows][:, :K // 2], oc)
    assert np.array_equal(unswizzle(g["sf"], rows[-1] + 1, K // 16, g["sf_cols"])[rows], os_)
    return ts


@pytest.mark.parametrize("M,K", [(64, 256), (3, 16), (130, 48), (257, 768), (40, 8192), (129, 2048)])
def test_quantize_and_scores_dense(L, M, K):
    x, _ = wl.activations(M, K, seed=M + K, n_outliers=max(1, K // 100), outlier_gain=20.0)
    g = _gpu_quant(L, x)
    ts = oracle.tensor_scale(x)
    amax, s_enc, s_dec, e = tscale_fields(g["ts"])
    assert (amax[0], s_enc[0], s_dec[0], e[0]) == (np.float32(ts.amax), np.float32(ts.s_enc), np.float32(ts.s_dec), ts.shift_e)
    oc, os_ = oracle.quantize(x, ts)
    assert np.array_equal(g["codes"][:, :K // 2], oc)
    assert np.array_equal(unswizzle(g["sf"], M, K // 16, g["sf_cols"]), os_)
    pad = unswizzle(g["sf"], M, g["sf_cols"], g["sf_cols"])[:, K // 16:]
    assert not pad.any(), "scale padding must be zero"
    assert np.array_equal(g["scores"][0], oracle.scores(x, ts))


def test_quantize_every_bf16_value_at_unit_block_scale(L):
    """Every finite bf16 value with |v| <= 6 in blocks whose amax is 6 (tensor amax 6, block
    scale 448, encode scale exactly 1): exercises the E2M1 rounding and sign handling of the
    conversion instruction on every input bit pattern, ties included."""
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = wl.bf16_bits_to_f32(allbits)
    keep = allbits[np.isfinite(v) & (np.abs(v) <= 6.0)]
    n_blocks = (keep.size + 14) // 15
    vals = np.zeros(n_blocks * 15, np.uint16)
    vals[:keep.size] = keep
    blocks = np.concatenate([np.full((n_blocks, 1), wl.to_bf16_bits(np.array([6.0]))[0], np.uint16),
                             vals.reshape(n_blocks, 15)], axis=1)
    cols = 256
    per_row = cols // 16
    n_rows = (n_blocks + per_row - 1) // per_row
    x = np.zeros((n_rows * per_row, 16), np.uint16)
    x[:n_blocks] = blocks
    x[n_blocks:, 0] = blocks[0, 0]
    x = x.reshape(n_rows, cols)
    g = _gpu_quant(L, x)
    ts = oracle.tensor_scale(x)
    assert ts.s_enc == 448.0
    oc, os_ = oracle.quantize(x, ts)
    assert np.all(os_ == 0x7E)
    assert np.array_equal(g["codes"][:, :cols // 2], oc)
    assert np.array_equal(unswizzle(g["sf"], n_rows, cols // 16, g["sf_cols"]), os_)
    assert np.array_equal(g["scores"][0], oracle.scores(x, ts))


def test_quantize_extreme_scales(L):
    """Tiny and huge tensors (block scales at the E4M3 subnormal end, scale splitting in the
    score), all-zero rows and a tensor of zeros."""
    rng = np.random.default_rng(0)
    for mag in [1e-30, 1e-8, 3e-3, 1e4, 1e30]:
        x = wl.to_bf16_bits(rng.standard_normal((33, 64)) * mag * (10.0 ** rng.uniform(-6, 0, (33, 64))))
        x[5] = 0
        g = _gpu_quant(L, x)
        ts = oracle.tensor_scale(x)
        oc, os_ = oracle.quantize(x, ts)
        assert np.array_equal(g["codes"][:, :32], oc), mag
        assert np.array_equal(unswizzle(g["sf"], 33, 4, g["sf_cols"]), os_), mag
        assert np.array_equal(g["scores"][0], oracle.scores(x, ts)), mag
    z = np.zeros((8, 32), np.uint16)
    g = _gpu_quant(L, z)
    assert not g["codes"][:, :16].any()
    assert tscale_fields(g["ts"])[1][0] == 1.0


@pytest.mark.parametrize("M,K,k", [(64, 256, 16), (200, 512, 64), (96, 768, 32), (50, 256, 256), (17, 4096, 64),
                                   (31, 6144, 128), (130, 768, 384), (40, 2048, 1024), (9, 4096, 4096),
                                   (64, 1024, 1024)])
@PATHS
def test_rac_select_and_tail_dense(L, M, K, k, tail_path):
    x, _ = wl.activations(M, K, seed=7 * M + K, n_outliers=max(2, K // 64), outlier_gain=16.0)
    g = _gpu_quant(L, x, k=k)
    q = oracle.rac_quantize(x, k)
    assert np.array_equal(g["scores"][0], q.scores)
    assert np.array_equal(g["idx"][0], q.idx)
    assert np.array_equal(g["codes"][:, :K // 2], q.codes)
    assert np.array_equal(g["codes"][:, K // 2:(K + k) // 2], q.tail_codes)
    sfl = unswizzle(g["sf"], M, g["sf_cols"], g["sf_cols"])
    assert np.array_equal(sfl[:, :K // 16], q.scales)
    assert np.array_equal(sfl[:, K // 16:(K + k) // 16], q.tail_scales)
    assert not sfl[:, (K + k) // 16:].any()


def test_topk_ties_and_degenerate(L):
    """Channels with equal scores (duplicated columns) are taken lowest index first; k = K."""
    x, _ = wl.activations(40, 256, seed=3, n_outliers=0)
    x[:, 128:] = x[:, :128]          # every score appears twice
    for k in [16, 48, 128, 256]:
        g = _gpu_quant(L, x, k=k)
        q = oracle.rac_quantize(x, k)
        assert np.array_equal(g["idx"][0], q.idx), k
        assert np.array_equal(g["codes"][:, 128:(256 + k) // 2], np.concatenate([q.codes[:, 128:], q.tail_codes], 1))
    z = np.zeros((16, 64), np.uint16)
    g = _gpu_quant(L, z, k=32)
    assert list(g["idx"][0]) == list(range(32))


@PATHS
def test_grouped_quantize_scores_and_tails(L, tail_path):
    """Row groups with padding gaps (the routed layout): per-group tensor scale, scores, S."""
    rng = np.random.default_rng(11)
    G, K, k = 6, 768, 32
    counts = [0, 5, 300, 128, 1, 77]
    off = [0]
    for c in counts:
        off.append(off[-1] + (c + 127) // 128 * 128)
    rows = off[-1]
    x, _ = wl.activations(rows, K, seed=5, n_outliers=8, outlier_gain=8.0)
    # make every group's magnitude different
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    for gi in range(G):
        xf[off[gi]:off[gi + 1]] *= 2.0 ** rng.integers(-5, 5)
    x = wl.to_bf16_bits(xf)
    g = _gpu_quant(L, x, k=k, groups=G, grp_off=off, grp_rows=counts)
    amax, s_enc, s_dec, e = tscale_fields(g["ts"])
    sfl = unswizzle(g["sf"], rows, g["sf_cols"], g["sf_cols"])
    for gi in range(G):
        a, c = off[gi], counts[gi]
        if c == 0:
            assert amax[gi] == 0 and s_enc[gi] == 1.0
            assert not g["scores"][gi].any()
            continue
        xs = x[a:a + c]
        q = oracle.rac_quantize(xs, k)
        assert amax[gi] == np.float32(q.ts.amax) and s_dec[gi] == np.float32(q.ts.s_dec)
        assert np.array_equal(g["scores"][gi], q.scores)
        assert np.array_equal(g["idx"][gi], q.idx)
        assert np.array_equal(g["codes"][a:a + c, :K // 2], q.codes)
        assert np.array_equal(g["codes"][a:a + c, K // 2:(K + k) // 2], q.tail_codes)
        assert np.array_equal(sfl[a:a + c, :K // 16], q.scales)
        assert np.array_equal(sfl[a:a + c, K // 16:(K + k) // 16], q.tail_scales)
        # rows of the padding gap are untouched
        assert np.all(g["codes"][a + c:off[gi + 1]] == 0xAB)


@pytest.mark.parametrize("G,N,K", [(1, 256, 256), (3, 128, 1536), (2, 384, 4160 - 64)])
def test_weight_qdq_matches_oracle_and_activation_quantizer(L, G, N, K):
    w = wl.weights((G, N, K), 0.02, seed=G * N + K)
    wt = bf16_tensor(w.reshape(G * N, K)).view(G, N, K)
    sf_cols = L.sf_cols(K)
    ld = (K // 2 + 15) // 16 * 16
    codes = torch.zeros(G * N, ld, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(L.sf_bytes(G * N, sf_cols), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(G, 4, dtype=torch.float32, device="cuda")
    what_b = torch.zeros(G * N, K, dtype=torch.bfloat16, device="cuda")
    what_f = torch.zeros(G * N, K, dtype=torch.float32, device="cuda")
    L.weight_qdq(wt, G, N, K, codes, sf, sf_cols, ts, w_hat=what_b, w_hat_dtype=L.NVQ_BF16)
    codes2 = torch.zeros_like(codes)
    sf2 = torch.zeros_like(sf)
    ts2 = torch.zeros_like(ts)
    L.weight_qdq(wt, G, N, K, codes2, sf2, sf_cols, ts2, w_hat=what_f, w_hat_dtype=L.NVQ_F32)
    torch.cuda.synchronize()
    assert torch.equal(codes, codes2) and torch.equal(sf, sf2)
    c = codes.cpu().numpy()
    sfl = unswizzle(sf, G * N, K // 16, sf_cols)
    _, _, s_dec, _ = tscale_fields(ts)
    for gi in range(G):
        wg = w[gi]
        t = oracle.tensor_scale(wg)
        oc, os_ = oracle.quantize(wg, t)
        assert np.array_equal(c[gi * N:(gi + 1) * N, :K // 2], oc)
        assert np.array_equal(sfl[gi * N:(gi + 1) * N], os_)
        assert s_dec[gi] == np.float32(t.s_dec)
        dq = oracle.dequantize(oc, os_, t.s_dec)
        assert np.array_equal(what_f[gi * N:(gi + 1) * N].cpu().numpy(), dq)
        assert np.array_equal(what_b[gi * N:(gi + 1) * N].cpu().view(torch.int16).numpy().view(np.uint16),
                              oracle.bf16_round(dq))
        # Eq. (16): the rollout activation quantizer on the same bytes gives the same codes
        g1 = _gpu_quant(L, wg)
        assert np.array_equal(g1["codes"][:, :K // 2], oc)
        assert np.array_equal(unswizzle(g1["sf"], N, K // 16, g1["sf_cols"]), os_)


def test_argument_errors_are_reported_before_launch(L):
    x = torch.zeros(4, 24, dtype=torch.bfloat16, device="cuda")
    codes = torch.zeros(4, 16, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(512, dtype=torch.uint8, device="cuda")
    ts = torch.zeros(1, 4, device="cuda")
    with pytest.raises(L.NvqError) as e:
        L.nvfp4_quantize(x, codes, sf, 4, ts)     # K = 24 is not a multiple of 16
    assert e.value.status == 2
    with pytest.raises(L.NvqError) as e:
        L.LIB and L.rac_select_quantize(torch.zeros(4, 32, dtype=torch.bfloat16, device="cuda"), ts,
                                        torch.zeros(32, dtype=torch.int64, device="cuda"), 8, codes, sf, 4,
                                        torch.zeros(8, dtype=torch.int32, device="cuda"))
    assert e.value.status == 2


@pytest.mark.parametrize("G,N,K,k,per_group", [(3, 384, 272, 32, True), (1, 256, 2048, 64, False),
                                               (2, 128, 16, 16, True), (4, 128, 1536, 48, True),
                                               (1, 128, 768, 400, False), (2, 128, 1536, 768, True),
                                               (1, 256, 256, 256, False)])
@PATHS
def test_weight_tail_channel_major_path(L, G, N, K, k, per_group, tail_path):
    """nvfp4_channel_major holds every code and scale of the weights at its channel-major place,
    and rac_weight_tail from that copy writes the same bytes as the row-major path and the oracle
    (ragged K: 272 = 17 blocks, 136 code bytes per row)."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import ChannelMajor, quantize_weights
    w = wl.weights((G, N, K), 0.02, seed=G + N + K + k)
    op = quantize_weights(bf16_tensor(w.reshape(G * N, K)).view(G, N, K), k)
    cm = ChannelMajor.of(op, G, N)
    rng = np.random.default_rng(K + k)
    idx_np = np.stack([np.sort(rng.choice(K, k, replace=False)) for _ in range(G if per_group else 1)]).astype(np.int32)
    idx = torch.from_numpy(idx_np).cuda()
    codes_rm, sf_rm = op.codes.clone(), op.sf.clone()
    L.rac_weight_tail(G, N, K, k, idx, codes_rm, sf_rm, op.sf_cols, op.tscale, idx_per_group=per_group)
    codes_cm, sf_cm = op.codes.clone(), op.sf.clone()
    L.rac_weight_tail(G, N, K, k, idx, codes_cm, sf_cm, op.sf_cols, op.tscale, idx_per_group=per_group,
                      cm_codes=cm.codes, cm_sf=cm.sf)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    # the copy: byte (g, j, m) = channel j of rows 2m | 2m+1; scale (g, c, n)
    c = op.codes.cpu().numpy()[:, :K // 2]
    nib = np.empty((G * N, K), np.uint8)
    nib[:, 0::2], nib[:, 1::2] = c & 0xF, c >> 4
    nib = nib.reshape(G, N, K).transpose(0, 2, 1)  # [G, K, N]
    assert np.array_equal(cm.codes.cpu().numpy(), nib[:, :, 0::2] | (nib[:, :, 1::2] << 4))
    sfl = unswizzle(op.sf, G * N, K // 16, op.sf_cols).reshape(G, N, K // 16).transpose(0, 2, 1)
    assert np.array_equal(cm.sf.cpu().numpy(), sfl)
    # both tail paths agree byte for byte, and with the oracle
    assert torch.equal(codes_rm, codes_cm) and torch.equal(sf_rm, sf_cm)
    tc_all = codes_cm.cpu().numpy()
    tsc_all = unswizzle(sf_cm, G * N, op.sf_cols, op.sf_cols)
    for g in range(G):
        wts = oracle.tensor_scale(w[g])
        wc, ws = oracle.quantize(w[g], wts)
        tc, tsc = oracle.weight_tail(wc, ws, wts, idx_np[g if per_group else 0])
        rows = slice(g * N, (g + 1) * N)
        assert np.array_equal(tc_all[rows, K // 2:(K + k) // 2], tc)
        assert np.array_equal(tsc_all[rows, K // 16:(K + k) // 16], tsc)
        assert not tsc_all[rows, (K + k) // 16:].any()


def test_quantize_with_given_amax_equals_measured(L):
    """amax_given: tscale[g].amax set by the caller (as the GEMM epilogue leaves it) gives the
    same tensor scales, codes, scales and scores as the call that measures amax itself."""
    counts = [200, 0, 129]
    off = [0, 256, 256, 512]
    K = 768
    x = np.zeros((512, K), np.uint16)
    for g, c in enumerate(counts):
        if c:
            xg, _ = wl.activations(c, K, seed=40 + g, n_outliers=8, outlier_gain=15.0)
            x[off[g]:off[g] + c] = xg
    a = _gpu_quant(L, x, groups=3, grp_off=off, grp_rows=counts)
    xt = bf16_tensor(x)
    ts = a["ts"].clone()
    ts[:, 1:] = 0.0  # only amax is given
    sf_cols = a["sf_cols"]
    codes = torch.full((512, a["codes"].shape[1]), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full_like(a["sf"], 0xCD)
    scores = torch.zeros(3, K, dtype=torch.int64, device="cuda")
    go = torch.tensor(off, dtype=torch.int64, device="cuda")
    gr = torch.tensor(counts, dtype=torch.int64, device="cuda")
    L.nvfp4_quantize(xt, codes, sf, sf_cols, ts, scores=scores, grp_off=go, grp_rows=gr, groups=3, zero_pad=True,
                     amax_given=True)
    torch.cuda.synchronize()
    assert torch.equal(ts.view(torch.int32), a["ts"].view(torch.int32))
    assert np.array_equal(codes.cpu().numpy(), a["codes"]) and torch.equal(sf, a["sf"])
    assert np.array_equal(scores.cpu().numpy().view(np.uint64), a["scores"])


@PATHS
def test_select_and_residual_tail_split_equals_combined(L, tail_path):
    """rac_select followed by rac_residual_tail writes exactly what rac_select_quantize writes."""
    counts = [300, 0, 129]
    off = [0, 384, 384, 640]
    K, k = 768, 32
    x = np.zeros((640, K), np.uint16)
    for g, c in enumerate(counts):
        if c:
            xg, _ = wl.activations(c, K, seed=60 + g, n_outliers=8, outlier_gain=15.0)
            x[off[g]:off[g] + c] = xg
    a = _gpu_quant(L, x, k=k, groups=3, grp_off=off, grp_rows=counts)
    xt = bf16_tensor(x)
    go = torch.tensor(off, dtype=torch.int64, device="cuda")
    gr = torch.tensor(counts, dtype=torch.int64, device="cuda")
    sf_cols = a["sf_cols"]
    codes = torch.full((640, a["codes"].shape[1]), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full_like(a["sf"], 0xCD)
    ts = torch.zeros(3, 4, dtype=torch.float32, device="cuda")
    scores = torch.zeros(3, K, dtype=torch.int64, device="cuda")
    L.nvfp4_quantize(xt, codes, sf, sf_cols, ts, scores=scores, grp_off=go, grp_rows=gr, groups=3)
    idx = torch.zeros(3, k, dtype=torch.int32, device="cuda")
    L.rac_select(scores, K, k, idx, groups=3)
    L.rac_residual_tail(xt, ts, idx, k, codes, sf, sf_cols, grp_off=go, grp_rows=gr, groups=3)
    torch.cuda.synchronize()
    assert np.array_equal(idx.cpu().numpy(), a["idx"])
    assert np.array_equal(codes.cpu().numpy(), a["codes"]) and torch.equal(sf, a["sf"])


@pytest.mark.parametrize("M,K,k", [(64, 256, 16), (130, 768, 0), (200, 1024, 128), (9, 512, 512), (257, 4096, 1024)])
def test_rac_reconstruct_dense(L, M, K, k):
    """X~ of Eq. (21) read back from the GPU operand equals the oracle's binary32 X~ bit for bit."""
    x, _ = wl.activations(M, K, seed=3 * M + k, n_outliers=max(1, K // 64), outlier_gain=20.0)
    g = _gpu_quant(L, x, k=k)
    out = torch.full((M, K), float("nan"), dtype=torch.float32, device="cuda")
    L.rac_reconstruct(g["codes_d"], g["sf"], g["sf_cols"], g["ts"], K, k, g["idx_d"] if k else None, out)
    torch.cuda.synchronize()
    ref = oracle.rac_reconstruct(oracle.rac_quantize(x, k))
    assert np.array_equal(out.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_rac_reconstruct_grouped_with_gaps(L):
    """Per-group tensor scales and channel sets, padding rows between groups left unwritten."""
    G, K, k = 4, 512, 64
    counts = [3, 0, 200, 129]
    off = [0]
    for c in counts:
        off.append(off[-1] + (c + 127) // 128 * 128)
    rows = off[-1]
    x, _ = wl.activations(rows, K, seed=8, n_outliers=6, outlier_gain=12.0)
    g = _gpu_quant(L, x, k=k, groups=G, grp_off=off, grp_rows=counts)
    out = torch.full((rows, K), -1.0, dtype=torch.float32, device="cuda")
    L.rac_reconstruct(g["codes_d"], g["sf"], g["sf_cols"], g["ts"], K, k, g["idx_d"], out, grp_off=g["go"],
                      grp_rows=g["gr"], groups=G)
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    for gi in range(G):
        a, c = off[gi], counts[gi]
        if c:
            ref = oracle.rac_reconstruct(oracle.rac_quantize(x[a:a + c], k))
            assert np.array_equal(o[a:a + c].view(np.uint32), ref.view(np.uint32))
        assert np.all(o[a + c:off[gi + 1]] == -1.0)
