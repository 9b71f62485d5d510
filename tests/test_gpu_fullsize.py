"""Parity at the full sizes of the five workloads, through the same calls and launch
configuration as the benchmark.  Everything the oracle can afford at full size is compared in
full (activation codes, scales, scores and selected channels); GEMM outputs are compared at
sampled positions, with the oracle fed the GPU operands only after those operands were
checked bit-exact against the oracle on the same rows."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import GEMM_RTOL, bf16_tensor, gemm_error, tscale_fields, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 32)
    return _lib


def test_activation_quantizer_rac_8192x4096_full(L):
    """Workload actquant_rac_8192x4096_k64: every code, scale, score and selected channel."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    cfg = wl.CFG_ACT
    x_bits, _, _ = cfg.make()
    M, K, k = cfg.M, cfg.K, cfg.k
    x = bf16_tensor(x_bits)
    op = Operand.empty(M, K, k)
    scores = torch.zeros(K, dtype=torch.int64, device="cuda")
    idx = torch.zeros(k, dtype=torch.int32, device="cuda")
    L.nvfp4_quantize(x, op.codes, op.sf, op.sf_cols, op.tscale, scores=scores)
    L.rac_select_quantize(x, op.tscale, scores, k, op.codes, op.sf, op.sf_cols, idx)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    q = oracle.rac_quantize(x_bits, k)
    amax, s_enc, s_dec, e = tscale_fields(op.tscale)
    assert (amax[0], s_dec[0], e[0]) == (np.float32(q.ts.amax), np.float32(q.ts.s_dec), q.ts.shift_e)
    assert np.array_equal(scores.cpu().numpy().view(np.uint64), q.scores)
    assert np.array_equal(idx.cpu().numpy(), q.idx)
    codes = op.codes.cpu().numpy()
    assert np.array_equal(codes[:, :K // 2], q.codes)
    assert np.array_equal(codes[:, K // 2:(K + k) // 2], q.tail_codes)
    sfl = unswizzle(op.sf, M, op.sf_cols, op.sf_cols)
    assert np.array_equal(sfl[:, :K // 16], q.scales)
    assert np.array_equal(sfl[:, K // 16:(K + k) // 16], q.tail_scales)


def test_dense_rac_linear_4096x4096x14336_sampled(L):
    """Workload dense_rac_gemm_4096x4096x14336_k64 through RacLinear (the benchmark's calls):
    activation operand on sampled rows and selection in full, weight operand on sampled rows,
    output at 2048 sampled positions."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import RacLinear
    cfg = wl.CFG_DENSE
    x_bits, w_bits, _ = cfg.make()
    M, K, N, k = cfg.M, cfg.K, cfg.N, cfg.k
    layer = RacLinear(bf16_tensor(w_bits), k, M)
    out = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    layer.forward(bf16_tensor(x_bits), out)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    rng = np.random.default_rng(12)
    ts = oracle.tensor_scale(x_bits)
    s = oracle.scores(x_bits, ts)
    idx = oracle.topk(s, k)
    assert np.array_equal(layer.idx.cpu().numpy(), idx)
    rows = np.sort(rng.choice(M, 64, replace=False))
    wrows = np.sort(rng.choice(N, 64, replace=False))
    xs = x_bits[rows]
    ac, asc = oracle.quantize(xs, ts)
    tc, tsc = oracle.rac_tail(xs, ts, idx)
    ga = layer.a.codes.cpu().numpy()[rows, :(K + k) // 2]
    gs = unswizzle(layer.a.sf, M, (K + k) // 16, layer.a.sf_cols)[rows]
    assert np.array_equal(ga, np.concatenate([ac, tc], 1)) and np.array_equal(gs, np.concatenate([asc, tsc], 1))
    wts = oracle.tensor_scale(w_bits)
    wc, ws = oracle.quantize(w_bits[wrows], wts)
    _, _, w_sdec, _ = tscale_fields(layer.w.tscale)
    assert w_sdec[0] == np.float32(wts.s_dec)
    gb = layer.w.codes.cpu().numpy()
    gbs = unswizzle(layer.w.sf, N, (K + k) // 16, layer.w.sf_cols)
    assert np.array_equal(gb[wrows, :K // 2], wc) and np.array_equal(gbs[wrows, :K // 16], ws)
    # weight tail on the sampled rows (built by the GEMM call from the checked stored weights)
    wtc, wtsc = oracle.weight_tail(gb[wrows, :K // 2], gbs[wrows, :K // 16], wts, idx)
    assert np.array_equal(gb[wrows, K // 2:(K + k) // 2], wtc) and np.array_equal(gbs[wrows, K // 16:(K + k) // 16], wtsc)
    mi = rng.integers(0, 64, 2048)
    ni = rng.integers(0, 64, 2048)
    ref = oracle.gemm_pairs(ga, gs, gb[wrows, :(K + k) // 2], gbs[wrows, :(K + k) // 16], ts.s_dec, wts.s_dec, mi, ni)
    y = out.float().cpu().numpy()[rows[mi], wrows[ni]]
    assert gemm_error(y, ref) <= GEMM_RTOL


@pytest.mark.parametrize("which", ["prefill", "decode"])
def test_moe_layer_fullsize_sampled(L, which):
    """The two MoE workloads at full size, stage-wise on sampled rows and experts."""
    from tests.test_gpu_moe import _check_layer
    c = wl.CFG_MOE_PREFILL if which == "prefill" else wl.CFG_MOE_DECODE
    wh, wy = _check_layer(L, T=c.T, H=c.H, E=c.E, topk=c.topk, I=c.I, k=c.k, routing=c.routing, seed=c.seed,
                          sample_rows=96, n_outliers=c.n_outliers, max_experts=6)
    assert wh <= GEMM_RTOL and wy <= GEMM_RTOL


def test_weight_qdq_all_experts_decode_workload(L):
    """Trainer-side QDQ of all 128 experts' W13 [128, 3072, 4096] and W2 [128, 4096, 1536]:
    codes and scales equal the rollout quantizer's (the activation-quantizer kernel on the same
    bytes, grouped per expert) for every expert, and the oracle on sampled experts and rows."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    c = wl.CFG_MOE_DECODE
    w13_bits, w2_bits = c.make_weights()
    rng = np.random.default_rng(5)
    for wb in (w13_bits, w2_bits):
        G, N, K = wb.shape
        w = bf16_tensor(wb.reshape(G * N, K))
        a = Operand.empty(G * N, K, 0, G)
        what = torch.empty(G * N, K, dtype=torch.bfloat16, device="cuda")
        L.weight_qdq(w.view(G, N, K), G, N, K, a.codes, a.sf, a.sf_cols, a.tscale, w_hat=what)
        b = Operand.empty(G * N, K, 0, G)
        go = torch.arange(0, G * N + 1, N, dtype=torch.int64, device="cuda")
        L.nvfp4_quantize(w, b.codes, b.sf, b.sf_cols, b.tscale, grp_off=go, groups=G, zero_pad=True)
        torch.cuda.synchronize()
        assert L.device_status() == (0, 0)
        # tensor-scale rows compared as raw bits (the int32 exponent field is not a float)
        assert torch.equal(a.codes, b.codes) and torch.equal(a.sf, b.sf)
        assert torch.equal(a.tscale.view(torch.int32), b.tscale.view(torch.int32))
        _, _, s_dec, _ = tscale_fields(a.tscale)
        for g in rng.choice(G, 3, replace=False):
            t = oracle.tensor_scale(wb[g])
            assert s_dec[g] == np.float32(t.s_dec)
            rows = np.sort(rng.choice(N, 32, replace=False))
            oc, os_ = oracle.quantize(wb[g][rows], t)
            assert np.array_equal(a.codes[g * N + rows].cpu().numpy()[:, :K // 2], oc)
            assert np.array_equal(unswizzle(a.sf, (g + 1) * N, K // 16, a.sf_cols)[g * N + rows], os_)
            dq = oracle.dequantize(oc, os_, t.s_dec)
            assert np.array_equal(what[g * N + rows].cpu().view(torch.int16).numpy().view(np.uint16), oracle.bf16_round(dq))
        del w, a, b, what
        torch.cuda.empty_cache()
