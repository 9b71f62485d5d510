"""The block scale's division by 6 (QUADS §2.2 "FP4": one E4M3 scale per 16-element block; the
scale is t = fl(fl(amax_b / 6) * S_enc) rounded to E4M3).  The quantizer forms fl(amax_b / 6)
without a division (a multiply and an FMA correction), so two checks pin it:

- the library's self-check runs every finite non-negative bf16 value through that form and
  through CUDA's IEEE division __fdiv_rn, and must find no difference;
- every finite non-negative bf16 value is made the amax of one 16-element block, in row groups
  whose tensor scales put t inside the E4M3 range, and the scale bytes and codes must equal the
  oracle's (plain C, IEEE division) bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.nvfp4_testutil import bf16_tensor, tscale_fields, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 31)
    return _lib


def test_division_by_six_matches_ieee_division_for_every_bf16(L):
    res = torch.zeros(2, dtype=torch.int32, device="cuda")
    L.check_block_scale_division(res)
    count, first = (int(v) for v in res.cpu().numpy().view(np.uint32))
    assert count == 0, f"{count} bf16 values differ, lowest pattern {first:#06x}"
    assert first == 0xFFFFFFFF


def _every_bf16_as_block_amax(seed=5, K=256, binades=8):
    """Rows of 16-element blocks; block i of group j has amax = the i-th finite non-negative bf16
    value whose exponent field lies in [binades*j, binades*(j+1)); the other 15 elements are
    that value times a uniform factor in (-1, 1), rounded to bf16 (so their magnitudes do not
    exceed it), and the amax sits at a varying position with a random sign."""
    rng = np.random.default_rng(seed)
    vals = np.arange(0x7F80, dtype=np.uint32).astype(np.uint16)  # 0x0000 .. 0x7f7f
    exp_field = vals >> 7
    bpr = K // 16
    rows_per_group = binades * 128 // bpr
    blocks, grp_off = [], [0]
    for j in range(0, 255, binades):
        v = vals[(exp_field >= j) & (exp_field < j + binades)]
        n = rows_per_group * bpr
        v = np.concatenate([v, np.full(n - v.size, v[0], np.uint16)])  # pad with a repeat
        amax = (v.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        u = rng.uniform(-1.0, 1.0, size=(n, 16))
        blk = oracle.bf16_round((amax[:, None] * u).astype(np.float32))
        pos = rng.integers(0, 16, size=n)
        sign = rng.integers(0, 2, size=n).astype(np.uint16) << 15
        blk[np.arange(n), pos] = v | sign
        blocks.append(blk.reshape(rows_per_group, K))
        grp_off.append(grp_off[-1] + rows_per_group)
    return np.concatenate(blocks), np.array(grp_off, np.int64)


def test_every_bf16_value_as_block_amax_matches_oracle(L):
    x_bits, grp_off = _every_bf16_as_block_amax()
    M, K = x_bits.shape
    G = grp_off.size - 1
    x = bf16_tensor(x_bits)
    sfc = L.sf_cols(K)
    codes = torch.zeros(M, K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(L.sf_bytes(M, sfc), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(G, 4, dtype=torch.float32, device="cuda")
    go = torch.from_numpy(grp_off).cuda()
    L.nvfp4_quantize(x, codes, sf, sfc, ts, grp_off=go, groups=G, zero_pad=True)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    g_codes = codes.cpu().numpy()
    g_sf = unswizzle(sf, M, K // 16, sfc)
    amax, s_enc, s_dec, e = tscale_fields(ts)
    in_range = 0
    for g in range(G):
        r0, r1 = int(grp_off[g]), int(grp_off[g + 1])
        xs = np.ascontiguousarray(x_bits[r0:r1])
        t = oracle.tensor_scale(xs)
        assert (amax[g], s_enc[g], s_dec[g], e[g]) == (np.float32(t.amax), np.float32(t.s_enc), np.float32(t.s_dec),
                                                       t.shift_e), g
        oc, os_ = oracle.quantize(xs, t)
        assert np.array_equal(g_sf[r0:r1], os_), f"scale bytes differ in group {g}"
        assert np.array_equal(g_codes[r0:r1], oc), f"codes differ in group {g}"
        in_range += int(np.count_nonzero((os_ > 0) & (os_ < 0x7E)))
    # the grouping does put most blocks' scales strictly inside the E4M3 range
    assert in_range > 0.9 * (M * K // 16) * (30 / 32)
