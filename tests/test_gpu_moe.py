"""Stage-wise GPU parity of the MoE expert layer with W4A4 + RAC in both expert GEMMs.

Each stage is compared with the oracle fed by the GPU's own (already checked) upstream output:
dispatch, token quantization and selection, gather (bit-exact); gate/up GEMM with SwiGLU
(2e-3 rule); per-expert quantization and selection of h (bit-exact); down GEMM with the routing
weight (2e-3 rule); combine (bit-exact)."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import GEMM_RTOL, bf16_bits, bf16_tensor, gemm_error, tscale_fields, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 31)
    return _lib


def _operand_rows(op, rows, ktot):
    rows = np.asarray(rows)
    codes = op.codes[torch.from_numpy(rows).to(op.codes.device)].cpu().numpy()[:, :ktot // 2]
    sfl = unswizzle(op.sf, int(rows.max()) + 1, ktot // 16, op.sf_cols)[rows]
    return codes, sfl


def _check_layer(L, T, H, E, topk, I, k, routing, seed, sample_rows=None, n_outliers=None, max_experts=None,
                 k2=None):
    """k / k2: compensated channels at the gate/up / down site (k2 defaults to k); sample_rows: routed rows checked in the gate/up GEMM (None: all); max_experts: experts
    checked in the gate/up and down stages (None: all)."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import MoERacLayer
    cfg = wl.MoELayer("t", T=T, H=H, E=E, topk=topk, I=I, k=k, seed=seed, routing=routing,
                      n_outliers=max(1, H // 100) if n_outliers is None else n_outliers)
    x_bits, ids, tw, _ = cfg.make_tokens()
    w13_bits, w2_bits = cfg.make_weights()
    dev = "cuda"
    w13 = bf16_tensor(w13_bits.reshape(E * 2 * I, H)).view(E, 2 * I, H)
    w2 = bf16_tensor(w2_bits.reshape(E * H, I)).view(E, H, I)
    k2 = k if k2 is None else k2
    layer = MoERacLayer(w13, w2, k, topk, T, k2=k2)
    x = bf16_tensor(x_bits)
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    layer.forward(x, torch.from_numpy(ids).to(dev), torch.from_numpy(tw).to(dev), out)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)

    # 1. dispatch
    grp_off = layer.grp_off.cpu().numpy()
    grp_rows = layer.grp_rows.cpu().numpy()
    row_src = layer.row_src.cpu().numpy()
    row_of = layer.row_of.cpu().numpy()
    row_w = layer.row_w.cpu().numpy()
    o_off, o_src = oracle.moe_dispatch(ids, E)
    assert np.array_equal(grp_rows, np.diff(o_off))
    assert np.all(grp_off[:-1] % 128 == 0)
    for g in range(E):
        seg = row_src[grp_off[g]:grp_off[g] + grp_rows[g]]
        assert np.array_equal(seg, o_src[o_off[g]:o_off[g + 1]])
        assert np.all(row_src[grp_off[g] + grp_rows[g]:grp_off[g + 1]] == -1)
    assert np.array_equal(row_src[row_of], np.arange(T * topk))
    assert np.array_equal(row_w[row_of], tw.ravel())

    # 2. token quantization + selection (one tensor scale and one channel set for all tokens)
    q1 = oracle.rac_quantize(x_bits, k)
    assert np.array_equal(layer.idx1.cpu().numpy()[:k], q1.idx)
    a1c, a1s = _operand_rows(layer.a_tok, np.arange(T), H + k)
    assert np.array_equal(a1c, np.concatenate([q1.codes, q1.tail_codes], 1))
    assert np.array_equal(a1s, np.concatenate([q1.scales, q1.tail_scales], 1))

    # experts checked in the GEMM stages: all, or a few (the largest, the smallest non-empty, random)
    nonempty = np.nonzero(grp_rows)[0]
    if max_experts is not None and nonempty.size > max_experts:
        by_size = nonempty[np.argsort(grp_rows[nonempty])]
        pick = [by_size[-1], by_size[0]] + list(np.random.default_rng(seed).choice(by_size[1:-1], max_experts - 2, replace=False))
        experts = np.array(sorted(set(int(e) for e in pick)))
    else:
        experts = nonempty

    # 3. gather into the routed layout
    routed = np.nonzero(row_src >= 0)[0]
    routed = routed[np.isin(np.searchsorted(grp_off, routed, side="right") - 1, experts)]
    if sample_rows is not None and routed.size > sample_rows:
        routed = np.sort(np.random.default_rng(seed).choice(routed, sample_rows, replace=False))
    tok_of = np.where(row_src >= 0, row_src // topk, 0)
    arc, ars = _operand_rows(layer.a_routed, routed, H + k)
    assert np.array_equal(arc, a1c[tok_of[routed]]) and np.array_equal(ars, a1s[tok_of[routed]])
    pad = np.nonzero(row_src < 0)[0][:64]
    if pad.size:
        pc, ps = _operand_rows(layer.a_routed, pad, H + k)
        assert not pc.any() and not ps.any()

    # weights as the GEMM saw them (tails rebuilt inside the calls): check them against the oracle
    _, _, w13_sdec, _ = tscale_fields(layer.w13.tscale)
    _, _, w2_sdec, _ = tscale_fields(layer.w2.tscale)
    h_gpu = bf16_bits(layer.h)
    worst_h = 0.0
    groups_of_rows = np.searchsorted(grp_off, routed, side="right") - 1
    for g in np.unique(groups_of_rows):
        rows_g = routed[groups_of_rows == g]
        wg = w13_bits[g]
        wts = oracle.tensor_scale(wg)
        assert np.float32(wts.s_dec) == w13_sdec[g]
        wc, ws = oracle.quantize(wg, wts)
        tc, tsc = oracle.weight_tail(wc, ws, wts, q1.idx)
        bc, bs = _operand_rows(layer.w13, np.arange(g * 2 * I, (g + 1) * 2 * I), H + k)
        assert np.array_equal(bc, np.concatenate([wc, tc], 1)) and np.array_equal(bs, np.concatenate([ws, tsc], 1))
        ac, as_ = _operand_rows(layer.a_routed, rows_g, H + k)
        ref = oracle.gemm(ac, as_, bc, bs, q1.ts.s_dec, wts.s_dec)
        href = oracle.swiglu(ref[:, :I], ref[:, I:]).reshape(len(rows_g), I)
        worst_h = max(worst_h, gemm_error(wl.bf16_bits_to_f32(h_gpu[rows_g]), href))
    assert worst_h <= GEMM_RTOL, worst_h

    # 4./5. per-expert quantization of the GPU's h, selection, down GEMM with routing weights
    a2_amax, _, a2_sdec, _ = tscale_fields(layer.a2.tscale)
    idx2 = layer.idx2.cpu().numpy()
    y_gpu = bf16_bits(layer.y)
    worst_y = 0.0
    for g in experts:
        c = int(grp_rows[g])
        rows_g = np.arange(grp_off[g], grp_off[g] + c)
        hq = oracle.rac_quantize(h_gpu[rows_g], k2)
        assert np.float32(hq.ts.amax) == a2_amax[g] and np.float32(hq.ts.s_dec) == a2_sdec[g]
        assert np.array_equal(idx2[g, :k2], hq.idx)
        ac, as_ = _operand_rows(layer.a2, rows_g, I + k2)
        assert np.array_equal(ac, np.concatenate([hq.codes, hq.tail_codes], 1))
        assert np.array_equal(as_, np.concatenate([hq.scales, hq.tail_scales], 1))
        if sample_rows is not None and c > 64:
            pick = np.sort(np.random.default_rng(g).choice(c, 64, replace=False))
        else:
            pick = np.arange(c)
        wg = w2_bits[g]
        wts = oracle.tensor_scale(wg)
        wc, ws = oracle.quantize(wg, wts)
        tc, tsc = oracle.weight_tail(wc, ws, wts, hq.idx)
        bc, bs = _operand_rows(layer.w2, np.arange(g * H, (g + 1) * H), I + k2)
        assert np.array_equal(bc, np.concatenate([wc, tc], 1)) and np.array_equal(bs, np.concatenate([ws, tsc], 1))
        ref = oracle.gemm(ac[pick], as_[pick], bc, bs, hq.ts.s_dec, wts.s_dec)
        ref = ref * row_w[rows_g[pick]][:, None].astype(np.float64)
        worst_y = max(worst_y, gemm_error(wl.bf16_bits_to_f32(y_gpu[rows_g[pick]]), ref))
    assert worst_y <= GEMM_RTOL, worst_y

    # 6. combine of the GPU's y, bit-exact
    out_bits = bf16_bits(out)
    tsel = np.arange(T) if sample_rows is None else np.sort(np.random.default_rng(1).choice(T, min(T, 512), replace=False))
    pos = row_of.reshape(T, topk)[tsel].ravel()
    ref_out = oracle.moe_combine(y_gpu, pos, topk)
    assert np.array_equal(out_bits[tsel], ref_out)
    return worst_h, worst_y


def test_moe_layer_small_zipf(L):
    _check_layer(L, T=300, H=256, E=8, topk=2, I=128, k=16, routing="zipf", seed=21)


def test_moe_layer_small_uniform_topk8(L):
    _check_layer(L, T=200, H=512, E=16, topk=8, I=256, k=32, routing="uniform", seed=22)


def test_moe_layer_without_rac(L):
    _check_layer(L, T=130, H=256, E=4, topk=2, I=128, k=0, routing="uniform", seed=23)


@pytest.mark.parametrize("k,k2", [(128, 64), (0, 32), (48, 0), (256, 128)])
def test_moe_layer_per_site_k(L, k, k2):
    """Different channel counts at the two sites, up to k = K at both (H = 256, I = 128)."""
    _check_layer(L, T=260, H=256, E=8, topk=2, I=128, k=k, k2=k2, routing="zipf", seed=24 + k + k2)


@pytest.mark.parametrize("use_graph", [True, False])
def test_host_pipeline_matches_direct_forward(L, use_graph):
    """HostPipeline (inputs copied up, forward, output copied back, neighbouring steps
    overlapped on three streams) returns exactly the layer's direct forward output."""
    from nvfp4_w4a4_quantized_quantize_gb300.layers import MoERacLayer
    from nvfp4_w4a4_quantized_quantize_gb300.pipeline import HostPipeline
    cfg = wl.MoELayer("t", T=200, H=256, E=8, topk=2, I=128, k=16, seed=31, routing="zipf", n_outliers=3)
    x_bits, ids, tw, _ = cfg.make_tokens()
    w13_bits, w2_bits = cfg.make_weights()
    layer = MoERacLayer(bf16_tensor(w13_bits.reshape(8 * 256, 256)).view(8, 256, 256),
                        bf16_tensor(w2_bits.reshape(8 * 256, 128)).view(8, 256, 128), 16, 2, 200)
    ref = torch.empty(200, 256, dtype=torch.bfloat16, device="cuda")
    layer.forward(bf16_tensor(x_bits), torch.from_numpy(ids).cuda(), torch.from_numpy(tw).cuda(), ref)
    torch.cuda.synchronize()
    pipe = HostPipeline(layer, 200, use_graph=use_graph)
    x_h = torch.from_numpy(x_bits.view(np.int16)).view(torch.bfloat16).pin_memory()
    out_h = torch.zeros(200, 256, dtype=torch.bfloat16).pin_memory()
    ms = pipe.run(x_h, torch.from_numpy(ids).pin_memory(), torch.from_numpy(tw).pin_memory(), out_h, 5)
    assert ms > 0 and L.device_status() == (0, 0)
    assert torch.equal(out_h.view(torch.int16), ref.cpu().view(torch.int16))


@pytest.mark.parametrize("topk,hidden", [(1, 264), (3, 2048), (8, 2048), (9, 520), (12, 64)])
def test_combine_slot_order_sum(L, topk, hidden):
    """moe_combine against the oracle's slot-order fp32 sum, for topk up to the kernel's
    all-loads-in-flight bound (8) and past it, with widths that leave threads idle.  Two pairs
    are left out (row_of = -1, as moe_dispatch marks an out-of-range expert id); the oracle sees
    those slots pointing at an all-zero row of y, which adds nothing."""
    T = 37
    n = T * topk
    rows = n + 6
    y_bits, _ = wl.activations(rows, hidden, seed=topk * 7 + hidden, n_outliers=2, outlier_gain=8.0)
    zero_row = rows - 1
    y_bits[zero_row] = 0
    rng = np.random.default_rng(topk)
    pos = rng.permutation(rows - 1)[:n].astype(np.int64)
    out_pairs = [2, (5 * topk + 1) % n]
    pos_gpu, pos_ref = pos.copy(), pos.copy()
    pos_gpu[out_pairs] = -1
    pos_ref[out_pairs] = zero_row
    out = torch.empty(T, hidden, dtype=torch.bfloat16, device="cuda")
    L.moe_combine(bf16_tensor(y_bits), torch.from_numpy(pos_gpu).cuda(), T, topk, hidden, out)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    assert np.array_equal(bf16_bits(out), oracle.moe_combine(y_bits, pos_ref, topk))
