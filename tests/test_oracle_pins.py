"""Pins of the CPU oracle to facts that do not come from the oracle itself.

Each test ties one part of the oracle to something fixed independently: a value printed in
QUADS (arXiv 2607.15810) §2.2 (the E2M1 grid, E4M3 with maximum 448), a hand-worked example,
a library routine (torch's float8_e4m3fn and bfloat16 casts, torch fp32 matmul), a closed form
or invariant of the method (odd symmetry, power-of-two scale invariance, Eq. (22)), or brute
force on small inputs.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _grid():
    with open(os.path.join(GOLDEN, "e2m1_grid.txt")) as f:
        line = [l for l in f if not l.startswith("#")][0]
    return [float(v) for v in line.split()]


def _f32_bits(a):
    return np.asarray(a, np.float32).view(np.uint32)


# ------------------------------------------------------------------------------ formats
def test_e2m1_decode_matches_printed_grid():
    grid = _grid()
    assert [oracle.e2m1_value(c) for c in range(8)] == grid
    assert [oracle.e2m1_value(8 | c) for c in range(8)] == [-g for g in grid]
    assert math.copysign(1.0, oracle.e2m1_value(8)) == -1.0


def test_e4m3_decode_matches_paper_and_torch():
    spec = dict(l.split() for l in open(os.path.join(GOLDEN, "e4m3_format.txt")) if not l.startswith("#"))
    vals = np.array([oracle.e4m3_value(b) for b in range(256)])
    finite = vals[np.isfinite(vals)]
    assert finite.max() == float(spec["max"])
    assert np.isnan(vals[0x7F]) and np.isnan(vals[0xFF])
    assert np.count_nonzero(np.isfinite(vals[:128])) == 127
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ok = np.isfinite(ref)
    assert np.array_equal(np.isfinite(vals), ok)
    assert np.array_equal(vals[ok], ref[ok])


def test_e4m3_encode_against_torch_cast():
    rng = np.random.default_rng(5)
    # every fp32 value that is an E4M3 midpoint or neighbour, plus random values over [0, 448]
    pos = np.array([oracle.e4m3_value(b) for b in range(0x7F)])
    mids = (pos[:-1] + pos[1:]) / 2
    t = np.concatenate([pos, mids, np.nextafter(mids, 0), np.nextafter(mids, 1000),
                        rng.uniform(0, 448, 20000), 2.0 ** rng.uniform(-14, 8.8, 20000)])
    t = t.astype(np.float32)
    t = t[t <= 448]
    got = oracle.e4m3_encode(t)
    ref = torch.from_numpy(t).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    # saturation (reading R3): above 448 -> 448
    big = np.array([448.0, 449.0, 464.0, 480.0, 1e6, 3e38], np.float32)
    assert np.all(oracle.e4m3_encode(big) == 0x7E)


def test_e2m1_encode_is_nearest_with_even_ties_exhaustive():
    grid = np.array(_grid())
    allbits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    v = wl.bf16_bits_to_f32(allbits)
    v = v[np.isfinite(v)]
    for scale in [1.0, 0.5, 2.0, 0.125, 3.0, 6.2222223, 1.7, 0.01]:
        with np.errstate(over="ignore"):
            y = (v * np.float32(scale)).astype(np.float32)
        y = y[np.isfinite(y)]
        c = oracle.e2m1_encode(y)
        a = np.abs(y.astype(np.float64))
        d = np.abs(a[:, None] - grid[None, :])
        best = d.min(axis=1)
        mag = c & 7
        assert np.all(d[np.arange(a.size), mag] == best), "not a nearest grid value"
        tie = (d == best[:, None]).sum(axis=1) > 1
        assert np.all(mag[tie] % 2 == 0), "tie not resolved to the even magnitude index"
        assert np.array_equal((c >> 3).astype(bool), np.signbit(y)), "sign bit not kept"


def test_e2m1_tie_examples():
    cases = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6), (7.0, 7),
             (1e9, 7), (-0.25, 8), (-5.0, 14), (0.0, 0), (-0.0, 8), (0.2499, 0), (0.2501, 1)]
    got = oracle.e2m1_encode(np.array([v for v, _ in cases], np.float32))
    assert [int(g) for g in got] == [c for _, c in cases]


def test_bf16_round_against_torch():
    rng = np.random.default_rng(1)
    f = np.concatenate([rng.standard_normal(50000) * 10.0 ** rng.uniform(-30, 30, 50000),
                        [0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0, 3e38]]).astype(np.float32)
    got = oracle.bf16_round(f)
    ref = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


# ------------------------------------------------------------------------------ quantizer
def test_hand_worked_block_example():
    ex = json.load(open(os.path.join(GOLDEN, "nvfp4_block_example.json")))
    x = wl.to_bf16_bits(np.array(ex["x"], np.float64))[None, :]
    assert np.array_equal(wl.bf16_bits_to_f32(x)[0], np.array(ex["x"], np.float32))
    ts = oracle.tensor_scale(x)
    assert ts.amax == ex["amax"] and ts.s_enc == ex["s_enc"]
    codes, scales = oracle.quantize(x, ts)
    assert [f"0x{b:02x}" for b in scales[0]] == ex["block_scale_bytes"]
    unpacked = np.stack([codes[0] & 15, codes[0] >> 4], axis=1).ravel()
    expect = np.array([int(c, 16) for blk in ex["codes"] for c in blk])
    assert np.array_equal(unpacked, expect)


def _rand_x(M, K, seed, outliers=3):
    x, _ = wl.activations(M, K, seed, "normal", 1.0, outliers, 16.0)
    return x


def test_round_trip_of_grid_values():
    grid = _grid()
    for j in [-8, -3, 0, 2, 5]:
        vals = np.array([g * 2.0 ** j for g in grid] + [-g * 2.0 ** j for g in grid])
        x = wl.to_bf16_bits(vals)[None, :]
        ts = oracle.tensor_scale(x)
        codes, scales = oracle.quantize(x, ts)
        dq = oracle.dequantize(codes, scales, ts.s_dec)[0]
        assert np.allclose(dq, vals, rtol=1e-6, atol=0)
        unpacked = np.stack([codes[0] & 15, codes[0] >> 4], axis=1).ravel()
        assert list(unpacked[:8]) == list(range(8))
        assert list(unpacked[8:]) == [8 | c for c in range(8)]


def test_saturation_and_scale_representability():
    x = _rand_x(64, 512, 3)
    ts = oracle.tensor_scale(x)
    codes, scales = oracle.quantize(x, ts)
    sv = np.array([oracle.e4m3_value(b) for b in range(256)])
    assert np.all(scales <= 0x7E), "every block scale is a finite non-negative E4M3 <= 448"
    dq = oracle.dequantize(codes, scales, ts.s_dec)
    d_b = (sv[scales].astype(np.float32) * np.float32(ts.s_dec)).astype(np.float32)
    assert np.all(np.abs(dq) <= 6.0 * np.repeat(d_b, 16, axis=1) * (1 + 1e-7))
    # the tensor amax maps to the top of the E4M3 x E2M1 range
    i, j = np.unravel_index(np.argmax(np.abs(wl.bf16_bits_to_f32(x))), x.shape)
    assert scales[i, j // 16] in (0x7E, 0x7D)


def test_power_of_two_scale_invariance():
    x = _rand_x(32, 256, 4)
    xf = wl.bf16_bits_to_f32(x)
    ts = oracle.tensor_scale(x)
    c0, s0 = oracle.quantize(x, ts)
    for j in [-6, -1, 1, 7]:
        x2 = wl.to_bf16_bits(xf.astype(np.float64) * 2.0 ** j)
        ts2 = oracle.tensor_scale(x2)
        c2, s2 = oracle.quantize(x2, ts2)
        assert np.array_equal(c0, c2) and np.array_equal(s0, s2)
        assert ts2.s_dec == np.float32(ts.s_dec * 2.0 ** j)


def test_odd_symmetry():
    x = _rand_x(32, 256, 5)
    xn = x ^ np.uint16(0x8000)
    ts = oracle.tensor_scale(x)
    c, s = oracle.quantize(x, ts)
    cn, sn = oracle.quantize(xn, oracle.tensor_scale(xn))
    assert np.array_equal(s, sn)
    assert np.array_equal(cn, c ^ np.uint8(0x88))


def test_block_encoding_is_nearest_for_the_block_scale():
    """Brute force: given each block's scale, every code is the nearest grid value of x * e_b,
    and the block scale is the E4M3 rounding of fl(amax_b / 6) * S_enc."""
    x = _rand_x(16, 128, 6)
    xf = wl.bf16_bits_to_f32(x)
    ts = oracle.tensor_scale(x)
    codes, scales = oracle.quantize(x, ts)
    grid = np.array(_grid())
    sv = np.array([oracle.e4m3_value(b) for b in range(256)])
    for i in range(16):
        for b in range(8):
            blk = xf[i, b * 16:(b + 1) * 16]
            t = np.float32(np.float32(np.abs(blk).max() / np.float32(6)) * np.float32(ts.s_enc))
            assert scales[i, b] == np.argmin(np.where(np.arange(256) <= 0x7E, np.abs(sv - float(t)), np.inf))
            e_b = np.float32(np.float32(ts.s_enc) / np.float32(sv[scales[i, b]]))
            y = (blk * e_b).astype(np.float32).astype(np.float64)
            cc = np.stack([codes[i] & 15, codes[i] >> 4], axis=1).ravel()[b * 16:(b + 1) * 16]
            got = np.array([oracle.e2m1_value(c) for c in cc])
            assert np.all(np.abs(np.abs(y) - np.abs(got)) <= np.min(np.abs(np.abs(y)[:, None] - grid[None, :]), axis=1))


def test_tensor_scale_edge_cases():
    z = np.zeros((4, 32), np.uint16)
    ts = oracle.tensor_scale(z)
    assert ts.s_enc == 1.0 and ts.s_dec == 1.0
    c, s = oracle.quantize(z, ts)
    assert not c.any() and not s.any()
    one = wl.to_bf16_bits(np.full((1, 16), 6.0))
    ts = oracle.tensor_scale(one)
    assert ts.s_enc == 448.0 and ts.shift_e == 4


def test_tiny_tensor_encode_factor_saturates_and_zeros_stay_signed_zeros():
    """Tensor amax below 2688 / FLT_MAX: S_enc is clamped to FLT_MAX (R4), and for a block scale
    below 1 the quotient fl(S_enc / sb) would overflow.  It saturates at FLT_MAX (R5), so every
    product x * e_b is finite: +0 and -0 encode as 0x0 and 0x8 (never as the code of a NaN,
    whose sign differs between hosts) and a non-zero x as the E2M1 of x * FLT_MAX."""
    fmax = np.float32(np.finfo(np.float32).max)
    v = 0x0080  # bf16 2^-126, the smallest normal
    x = np.array([[v, 0x0000, 0x8000, v | 0x8000] + [0x0000] * 12], np.uint16)
    ts = oracle.tensor_scale(x)
    assert ts.s_enc == fmax
    t = np.float32(np.float32(2.0 ** -126) / np.float32(6.0)) * fmax
    sb = oracle.e4m3_encode(np.array([t], np.float32))[0]
    assert 0 < oracle.e4m3_value(int(sb)) < 1.0   # the quotient S_enc / sb overflows binary32
    c, s = oracle.quantize(x, ts)
    assert s[0, 0] == sb
    codes = [(c[0, i // 2] >> (4 * (i % 2))) & 0xF for i in range(16)]
    big = oracle.e2m1_encode(np.array([np.float32(2.0 ** -126) * fmax], np.float32))[0]
    assert codes[:4] == [big, 0x0, 0x8, big | 0x8]
    assert codes[4:] == [0x0] * 12


# ------------------------------------------------------------------------------ RAC
def test_scores_rank_like_l2_norm():
    """Eq. (23): the integer score ranks channels as the L2 norm of the residual does."""
    for seed in range(3):
        x = _rand_x(96, 256, 10 + seed, outliers=5)
        ts = oracle.tensor_scale(x)
        s = oracle.scores(x, ts)
        r = oracle.residual(x, ts).astype(np.float64)
        l2sq = (r * r).sum(axis=0)
        # |q - |r| 2^(20-E)| <= 1/2 per element bounds the gap to the scaled L2 norm
        scale = 2.0 ** (20 - ts.shift_e)
        exact = l2sq * scale * scale
        bound = (np.abs(r).sum(axis=0) * scale + 0.25 * 96)
        assert np.all(np.abs(s.astype(np.float64) - exact) <= bound + 1e-9 * exact)
        eps = 2 * bound.max() / scale ** 2
        o_int = np.lexsort((np.arange(256), -s.astype(np.float64)))
        for a, b in zip(o_int[:-1], o_int[1:]):
            assert l2sq[a] >= l2sq[b] - eps


def test_residual_definition_sign():
    x = _rand_x(8, 64, 20)
    ts = oracle.tensor_scale(x)
    r = oracle.residual(x, ts)
    codes, scales = oracle.quantize(x, ts)
    dq = oracle.dequantize(codes, scales, ts.s_dec)
    assert np.array_equal(r, (wl.bf16_bits_to_f32(x) - dq).astype(np.float32))


def test_topk_against_brute_force_sort():
    rng = np.random.default_rng(7)
    for n, k in [(64, 16), (256, 64), (4096, 64), (300, 300)]:
        s = rng.integers(0, 50, n).astype(np.uint64) * np.uint64(1 << 40)  # many ties
        idx = oracle.topk(s, k)
        order = sorted(range(n), key=lambda j: (-int(s[j]), j))[:k]
        assert list(idx) == sorted(order)


def _reconstruct(x, q: "oracle.RacQuant"):
    return oracle.rac_reconstruct(q).astype(np.float64)


def test_rac_reconstruct_properties():
    """X-tilde (Eq. (21)): k = 0 is plain DQ(Q(X)); channels outside S keep DQ(Q(X)) bit for
    bit; on S every element is at least as close to X as DQ(Q(X)) (E2M1 rounding is to the
    nearest grid value and 0 is on the grid, so |R - DQ(Q(R))| <= |R|), up to the half ulp of
    the binary32 sum; and that sum is the correctly rounded fp64 sum of the two parts."""
    x = _rand_x(48, 384, 34, outliers=6)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    q0 = oracle.rac_quantize(x, 0)
    dq = oracle.dequantize(q0.codes, q0.scales, q0.ts.s_dec)
    assert np.array_equal(oracle.rac_reconstruct(q0).view(np.uint32), dq.view(np.uint32))
    for k in (16, 96, 384):
        q = oracle.rac_quantize(x, k)
        xt = oracle.rac_reconstruct(q)
        rest = np.setdiff1d(np.arange(384), q.idx)
        assert np.array_equal(xt[:, rest].view(np.uint32), dq[:, rest].view(np.uint32))
        sel = xt[:, q.idx].astype(np.float64)
        half_ulp = np.spacing(np.abs(xt[:, q.idx])).astype(np.float64) / 2
        assert np.all(np.abs(xf[:, q.idx] - sel) <= np.abs(xf[:, q.idx] - dq[:, q.idx]) + half_ulp)
        tail = oracle.dequantize(q.tail_codes, q.tail_scales, q.ts.s_dec).astype(np.float64)
        exact = dq[:, q.idx].astype(np.float64) + tail
        assert np.array_equal(sel.astype(np.float32), exact.astype(np.float32))
        # the compensation is not a no-op: some selected element moved
        assert np.any(xt[:, q.idx] != dq[:, q.idx])


def test_rac_reduces_activation_error_eq22_and_monotone_in_k():
    x = _rand_x(64, 512, 30, outliers=8)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    errs = []
    for k in [0, 16, 64, 256, 512]:
        q = oracle.rac_quantize(x, k)
        errs.append(np.linalg.norm(_reconstruct(x, q) - xf))
        if k:
            assert q.tail_codes.any()
            # selected channels are the k largest scores
            assert set(q.idx) == set(np.lexsort((np.arange(512), -q.scores.astype(np.float64)))[:k])
    assert errs[1] < errs[0], "Eq. (22): compensation must shrink the activation error"
    assert all(a > b for a, b in zip(errs[:-1], errs[1:])), errs


def test_rac_tail_equals_quantized_residual_on_selected_channels():
    x = _rand_x(16, 256, 31)
    q = oracle.rac_quantize(x, 32)
    r = oracle.residual(x, q.ts)
    rs = r[:, q.idx]
    dt = oracle.dequantize(q.tail_codes, q.tail_scales, q.ts.s_dec)
    # second-pass error never exceeds the residual it compensates (norm over each row)
    assert np.all(np.linalg.norm(rs - dt, axis=1) <= np.linalg.norm(rs, axis=1) + 1e-12)
    # odd symmetry: Q(-R) is the sign-flipped Q(R), so adding DQ(Q(R)) is Eq. (21)'s subtraction
    for i in range(16):
        c, sb = oracle.quantize_block16(-rs[i, :16], q.ts.s_enc)
        c2, sb2 = oracle.quantize_block16(rs[i, :16], q.ts.s_enc)
        assert sb == sb2 and np.array_equal(c, c2 ^ 8)


def test_k_equal_K_selects_every_channel():
    x = _rand_x(8, 64, 32)
    q = oracle.rac_quantize(x, 64)
    assert list(q.idx) == list(range(64))


def test_weight_tail_requantizes_dequantized_weights():
    w = wl.weights((32, 128), 0.02, 33)
    wts = oracle.tensor_scale(w)
    wc, ws = oracle.quantize(w, wts)
    idx = np.arange(0, 128, 4, dtype=np.int32)[:32]
    tc, tsc = oracle.weight_tail(wc, ws, wts, idx)
    wdq = oracle.dequantize(wc, ws, wts.s_dec)[:, idx]
    tdq = oracle.dequantize(tc, tsc, wts.s_dec)
    assert np.max(np.abs(tdq - wdq)) <= np.max(np.abs(wdq)) / 4  # within half a grid step of 6 -> 4
    # selecting a whole original block that keeps its amax reproduces it exactly
    idx2 = np.arange(16, 48, dtype=np.int32)
    tc2, tsc2 = oracle.weight_tail(wc, ws, wts, idx2)
    assert np.array_equal(oracle.dequantize(tc2, tsc2, wts.s_dec), oracle.dequantize(wc, ws, wts.s_dec)[:, 16:48])


# ------------------------------------------------------------------------------ GEMM
def test_gemm_exact_form_matches_fp64_and_torch():
    x = _rand_x(24, 160, 40)
    w = wl.weights((40, 160), 0.02, 41)
    tx, tw = oracle.tensor_scale(x), oracle.tensor_scale(w)
    ac, as_ = oracle.quantize(x, tx)
    bc, bs = oracle.quantize(w, tw)
    y = oracle.gemm(ac, as_, bc, bs, tx.s_dec, tw.s_dec)
    mi, ni = np.meshgrid(np.arange(24), np.arange(40), indexing="ij")
    y64 = oracle.gemm_pairs_fp64(ac, as_, bc, bs, tx.s_dec, tw.s_dec, mi.ravel(), ni.ravel()).reshape(24, 40)
    assert np.allclose(y, y64, rtol=1e-12, atol=1e-300)
    a = torch.from_numpy(oracle.dequantize(ac, as_, tx.s_dec))
    b = torch.from_numpy(oracle.dequantize(bc, bs, tw.s_dec))
    yt = (a @ b.T).numpy().astype(np.float64)
    assert np.allclose(y, yt, rtol=1e-4, atol=1e-5 * np.abs(y).max())


def test_gemm_tiny_brute_force():
    """M = 2, N = 3, K = 32: every term written out from the decoded codes and scales."""
    x = _rand_x(2, 32, 42, outliers=1)
    w = wl.weights((3, 32), 0.02, 43)
    tx, tw = oracle.tensor_scale(x), oracle.tensor_scale(w)
    ac, as_ = oracle.quantize(x, tx)
    bc, bs = oracle.quantize(w, tw)
    y = oracle.gemm(ac, as_, bc, bs, tx.s_dec, tw.s_dec)
    from fractions import Fraction as F
    for m in range(2):
        for n in range(3):
            tot = F(0)
            for c in range(32):
                ca = (ac[m, c // 2] >> (4 * (c % 2))) & 15
                cb = (bc[n, c // 2] >> (4 * (c % 2))) & 15
                tot += (F(oracle.e2m1_value(ca)) * F(oracle.e4m3_value(as_[m, c // 16]))
                        * F(oracle.e2m1_value(cb)) * F(oracle.e4m3_value(bs[n, c // 16])))
            ref = float(tot * F(float(tx.s_dec)) * F(float(tw.s_dec)))
            assert y[m, n] == pytest.approx(ref, rel=1e-15, abs=1e-300)


def test_gemm_transposed_operands_differ():
    """A plain check that the oracle does not silently symmetrise the operands."""
    x = _rand_x(16, 64, 44)
    tx = oracle.tensor_scale(x)
    ac, as_ = oracle.quantize(x, tx)
    y = oracle.gemm(ac, as_, ac[:8], as_[:8], tx.s_dec, tx.s_dec)
    assert y.shape == (16, 8)
    assert np.allclose(y[:8, :8], y[:8, :8].T)   # X X^T is symmetric...
    assert not np.allclose(y[8:, :], 0)


# ------------------------------------------------------------------------------ MoE plumbing
def test_dispatch_is_stable_counting_sort():
    ids, _ = wl.routing_zipf(257, 16, 4, 1.1, 9)
    grp_off, row_src = oracle.moe_dispatch(ids, 16)
    flat = ids.ravel()
    order = np.argsort(flat, kind="stable")
    assert np.array_equal(row_src, order.astype(np.int32))
    assert np.array_equal(grp_off, np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=16))]))


def test_swiglu_and_combine_against_torch():
    g = np.linspace(-8, 8, 101)
    u = np.linspace(2, -3, 101)
    ref = (torch.nn.functional.silu(torch.from_numpy(g)) * torch.from_numpy(u)).numpy()
    assert np.allclose(oracle.swiglu(g, u), ref, rtol=1e-14, atol=1e-300)
    rng = np.random.default_rng(3)
    y = wl.to_bf16_bits(rng.standard_normal((40, 24)))
    pos = rng.permutation(40).astype(np.int64)
    out = oracle.moe_combine(y, pos, 4)
    yt = torch.from_numpy(wl.bf16_bits_to_f32(y))[torch.from_numpy(pos)].view(10, 4, 24)
    acc = yt[:, 0].clone()
    for s in range(1, 4):
        acc = acc + yt[:, s]
    ref = acc.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(out, ref)


# ---------------------------------------------------------------- FP8 W8A8 baseline (readings R16-R18)
def test_fp8_encode_matches_torch_float8_on_every_bf16_value():
    """Reading R18's E4M3 rounding (nearest, ties to even, sign kept) against torch's own
    float8_e4m3fn conversion, for every finite bf16 value of magnitude <= 448."""
    import torch
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        v = wl.bf16_bits_to_f32(bits).astype(np.float64)
    ok = np.isfinite(v) & (np.abs(v) <= 448.0)
    v = v[ok]
    ours = np.array([oracle.lib().oracle_fp8_encode(float(t)) for t in v], np.uint8)
    ref = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def test_fp8_scale_exponent_closed_form():
    """Reading R17: e = max(-127, ceil(log2(amax / 448))), computed with exact rationals, on
    random and boundary magnitudes."""
    import math
    rng = np.random.default_rng(40)
    vals = list(np.exp(rng.uniform(-90, 90, 2000)))
    for k in range(-130, 128, 7):
        b = math.ldexp(448.0, k)
        vals += [b, np.nextafter(b, 0), np.nextafter(b, np.inf)]
    vals += [1e-45, 5e-40, 448.0, 449.0, 3.0e38]
    from fractions import Fraction
    for a in vals:
        # ceil(log2(a / 448)) by exact rational comparison with powers of two
        q = Fraction(float(a)) / 448
        c = math.ceil(math.log2(q))
        while Fraction(2) ** c < q:
            c += 1
        while Fraction(2) ** (c - 1) >= q:
            c -= 1
        assert oracle.fp8_scale_exponent(a) == max(-127, min(127, c)), a
    assert oracle.fp8_scale_exponent(0.0) == -127


def test_fp8_tiles_scale_independently_and_round_trip_within_e4m3_bound():
    """1 x 128 activation tiles and 128 x 128 weight tiles (reading R16): scaling one tile by a
    power of two changes only its scale byte, by that power, and none of the codes; every
    element dequantizes within half an E4M3 step of its value (relative 2^-4 in the normal
    range, absolute 2^(e-10) below it); ragged edges form partial tiles."""
    x = _rand_x(5, 300, 41, outliers=3)  # 300 = 2 x 128 + 44
    c, s = oracle.fp8_quantize(x, 1)
    assert s.shape == (5, 3)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    x2 = xf.copy()
    x2[3, 128:256] *= 2.0 ** 5
    c2, s2 = oracle.fp8_quantize(wl.to_bf16_bits(x2), 1)
    assert np.array_equal(c, c2)
    d = s2.astype(int) - s.astype(int)
    assert d[3, 1] == 5 and np.count_nonzero(d) == 1
    dq = oracle.fp8_dequantize(c, s, 1)
    e = np.repeat(s.astype(np.int64) - 127, 128, axis=1)[:, :300]
    scaled = np.abs(xf) * 2.0 ** (-e)
    err = np.abs(dq - xf) * 2.0 ** (-e)
    normal = scaled >= 2.0 ** -6
    assert np.all(err[normal] <= scaled[normal] * 2.0 ** -4)
    assert np.all(err[~normal] <= 2.0 ** -10)
    # the tile maximum maps to at most 448 and above 224 (the scale is the smallest power)
    for i in range(5):
        for t in range(3):
            m = np.abs(xf[i, 128 * t:128 * (t + 1)]).max()
            if m > 0:
                assert 224.0 < m * 2.0 ** (127 - int(s[i, t])) <= 448.0
    # weights: 128 x 128 tiles; an outlier in one tile leaves the others' scales alone
    w = wl.weights((256, 256), 0.02, 42)
    wc, ws = oracle.fp8_quantize(w, 128)
    wf = wl.bf16_bits_to_f32(w).astype(np.float64)
    wf[200, 30] = 50.0
    wc2, ws2 = oracle.fp8_quantize(wl.to_bf16_bits(wf), 128)
    assert ws.shape == (2, 2) and ws2[1, 0] > ws[1, 0]
    assert ws2[0, 0] == ws[0, 0] and ws2[0, 1] == ws[0, 1] and ws2[1, 1] == ws[1, 1]


def test_fp8_gemm_against_torch_float8_decode():
    """fp8_gemm against the same product with torch's float8_e4m3fn decoding of the codes."""
    import torch
    x = _rand_x(40, 384, 43, outliers=4)
    w = wl.weights((136, 384), 0.02, 44)
    ac, asc = oracle.fp8_quantize(x, 1)
    bc, bsc = oracle.fp8_quantize(w, 128)
    dec = lambda c: torch.from_numpy(c).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    a = dec(ac) * np.exp2(np.repeat(asc.astype(np.float64) - 127, 128, axis=1))
    b = dec(bc) * np.exp2(np.repeat(np.repeat(bsc.astype(np.float64) - 127, 128, axis=0)[:136], 128, axis=1))
    assert np.allclose(oracle.fp8_gemm(ac, asc, bc, bsc), a @ b.T, rtol=1e-12, atol=0)


def test_fp8_hand_worked_tiles():
    """The FP8 oracle against a row quantized by hand from readings R16-R18
    (tests/golden/fp8_tile_example.json: a full tile and an edge tile, signed zeros, a value
    that flushes to zero, and a scale below one)."""
    ex = json.load(open(os.path.join(GOLDEN, "fp8_tile_example.json")))
    x = np.zeros((1, ex["cols"]), np.float64)
    for j, v in ex["nonzero_x"].items():
        x[0, int(j)] = -0.0 if v == "-0" else v
    codes, scales = oracle.fp8_quantize(wl.to_bf16_bits(x), 1)
    assert list(scales[0]) == ex["scale_bytes"]
    want = np.zeros(ex["cols"], np.uint8)
    for j, c in ex["codes_nonzero"].items():
        want[int(j)] = c
    assert np.array_equal(codes[0], want)
