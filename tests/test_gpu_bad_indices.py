"""Caller-supplied indices outside their range, run for real.

The tails' channel lists (idx), the gather's row map (row_src), the reconstruction's channel
list and the dispatch's expert ids come from the caller.  Each kernel that reads one checks it
before any load or store through it: an index outside its range is recorded in the device
status word as NVQ_ERR_ARG, with the check's code in `where`, and replaced by an in-range value
(channel 0, a padding row, or the pair left out of the routing).  The output of such a call is
meaningless, and the status says so.  Every access stays inside the operands, so no GPU fault
is possible.  Each test reads the status back through nvq_device_status (which clears it), then
checks that the next call with valid indices is clean and exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import bf16_tensor, unswizzle

pytestmark = pytest.mark.gpu

ERR_ARG = 1
WHERE_EXPERT_ID, WHERE_CH_ACT, WHERE_CH_WEIGHT, WHERE_CH_RECON, WHERE_SRC_ROW = 41, 42, 43, 44, 45


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 31)
    assert _lib.device_status() == (0, 0)
    yield _lib
    _lib.set_tail_path(_lib.NVQ_TAIL_AUTO)


def _idx(values):
    return torch.tensor(np.asarray(values, dtype=np.int32), device="cuda")


@pytest.mark.parametrize("path", ["gather", "rows"])
def test_residual_tail_channel_outside_K(L, path):
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    M, K, k = 300, 256, 32
    x_bits, _ = wl.activations(M, K, seed=5, n_outliers=4, outlier_gain=10.0)
    x = bf16_tensor(x_bits)
    q = oracle.rac_quantize(x_bits, k)
    op = Operand.empty(M, K, k)
    L.nvfp4_quantize(x, op.codes, op.sf, op.sf_cols, op.tscale)
    bad = q.idx.copy()
    bad[3], bad[7] = K + 5, -1
    L.set_tail_path(L.NVQ_TAIL_GATHER if path == "gather" else L.NVQ_TAIL_ROWS)
    try:
        L.rac_residual_tail(x, op.tscale, _idx(bad), k, op.codes, op.sf, op.sf_cols)
        assert L.device_status() == (ERR_ARG, WHERE_CH_ACT)
        L.rac_residual_tail(x, op.tscale, _idx(q.idx), k, op.codes, op.sf, op.sf_cols)
        assert L.device_status() == (0, 0)
    finally:
        L.set_tail_path(L.NVQ_TAIL_AUTO)
    assert np.array_equal(op.codes.cpu().numpy()[:, K // 2:(K + k) // 2], q.tail_codes)
    sfl = unswizzle(op.sf, M, (K + k) // 16, op.sf_cols)
    assert np.array_equal(sfl[:, K // 16:], q.tail_scales)


@pytest.mark.parametrize("path", ["gather", "channel_major", "rows"])
def test_weight_tail_channel_outside_K(L, path):
    from nvfp4_w4a4_quantized_quantize_gb300.layers import ChannelMajor, quantize_weights
    G, N, K, k = 2, 128, 256, 32
    w_bits = wl.weights((G * N, K), 0.02, seed=91)
    op = quantize_weights(bf16_tensor(w_bits).view(G, N, K), k)
    idx = np.sort(np.random.default_rng(3).choice(K, k, replace=False)).astype(np.int32)
    bad = idx.copy()
    bad[5] = 1 << 20
    cm = ChannelMajor.of(op, G, N) if path == "channel_major" else None
    cm_args = dict(cm_codes=cm.codes, cm_sf=cm.sf) if cm is not None else {}
    L.set_tail_path(L.NVQ_TAIL_ROWS if path == "rows" else L.NVQ_TAIL_GATHER)
    try:
        L.rac_weight_tail(G, N, K, k, _idx(bad), op.codes, op.sf, op.sf_cols, op.tscale, **cm_args)
        assert L.device_status() == (ERR_ARG, WHERE_CH_WEIGHT)
        L.rac_weight_tail(G, N, K, k, _idx(idx), op.codes, op.sf, op.sf_cols, op.tscale, **cm_args)
        assert L.device_status() == (0, 0)
    finally:
        L.set_tail_path(L.NVQ_TAIL_AUTO)
    codes = op.codes.cpu().numpy()
    sfl = unswizzle(op.sf, G * N, (K + k) // 16, op.sf_cols)
    for g in range(G):
        wg = w_bits[g * N:(g + 1) * N]
        wts = oracle.tensor_scale(wg)
        wc, ws = oracle.quantize(wg, wts)
        tc, tsc = oracle.weight_tail(wc, ws, wts, idx)
        assert np.array_equal(codes[g * N:(g + 1) * N, K // 2:(K + k) // 2], tc)
        assert np.array_equal(sfl[g * N:(g + 1) * N, K // 16:], tsc)


def test_reconstruct_channel_outside_K(L):
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    M, K, k = 200, 256, 32
    x_bits, _ = wl.activations(M, K, seed=8, n_outliers=3, outlier_gain=10.0)
    x = bf16_tensor(x_bits)
    op = Operand.empty(M, K, k)
    sc = torch.zeros(K, dtype=torch.int64, device="cuda")
    idx = torch.zeros(k, dtype=torch.int32, device="cuda")
    L.nvfp4_quantize(x, op.codes, op.sf, op.sf_cols, op.tscale, scores=sc)
    L.rac_select_quantize(x, op.tscale, sc, k, op.codes, op.sf, op.sf_cols, idx)
    ref = torch.zeros(M, K, dtype=torch.float32, device="cuda")
    L.rac_reconstruct(op.codes, op.sf, op.sf_cols, op.tscale, K, k, idx, ref)
    assert L.device_status() == (0, 0)
    bad = idx.clone()
    bad[0] = K
    out = torch.zeros(M, K, dtype=torch.float32, device="cuda")
    L.rac_reconstruct(op.codes, op.sf, op.sf_cols, op.tscale, K, k, bad, out)
    assert L.device_status() == (ERR_ARG, WHERE_CH_RECON)
    L.rac_reconstruct(op.codes, op.sf, op.sf_cols, op.tscale, K, k, idx, out)
    assert L.device_status() == (0, 0)
    assert torch.equal(out, ref)


def test_gather_source_row_outside_the_source(L):
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    T, topk, H, k = 100, 2, 256, 32
    x_bits, _ = wl.activations(T, H, seed=9, n_outliers=3, outlier_gain=10.0)
    tok = Operand.empty(T, H, k)
    L.nvfp4_quantize(bf16_tensor(x_bits), tok.codes, tok.sf, tok.sf_cols, tok.tscale)
    cap = 256
    rs = np.full(cap, -1, np.int32)
    rs[:T * topk] = np.arange(T * topk)
    bad = rs.copy()
    bad[5] = T * topk + 3          # token row 101: beyond the 100 source rows
    out = Operand.empty(cap, H, k)
    out.codes.fill_(0x55)
    L.nvfp4_gather_rows(tok.codes, tok.sf, tok.sf_cols, T, _idx(bad), topk, H + k, out.codes, out.sf)
    assert L.device_status() == (ERR_ARG, WHERE_SRC_ROW)
    assert not out.codes[5, :(H + k) // 2].any()    # left as a padding row
    L.nvfp4_gather_rows(tok.codes, tok.sf, tok.sf_cols, T, _idx(rs), topk, H + k, out.codes, out.sf)
    assert L.device_status() == (0, 0)
    src = rs[:T * topk] // topk
    w = (H + k) // 2
    assert np.array_equal(out.codes.cpu().numpy()[:T * topk, :w], tok.codes.cpu().numpy()[src, :w])
    so = unswizzle(out.sf, cap, (H + k) // 16, out.sf_cols)
    st = unswizzle(tok.sf, T, (H + k) // 16, tok.sf_cols)
    assert np.array_equal(so[:T * topk], st[src]) and not so[T * topk:].any()


def test_dispatch_expert_id_outside_the_groups(L):
    T, topk, E = 64, 2, 8
    rng = np.random.default_rng(12)
    ids = rng.integers(0, E, size=(T, topk)).astype(np.int32)
    ids[3, 1], ids[10, 0] = E, -2
    w = rng.uniform(0.1, 1.0, size=(T, topk)).astype(np.float32)
    cap = L.moe_capacity(T, topk, E)
    dev = "cuda"
    grp_off = torch.zeros(E + 1, dtype=torch.int64, device=dev)
    grp_rows = torch.zeros(E, dtype=torch.int64, device=dev)
    row_src = torch.zeros(cap, dtype=torch.int32, device=dev)
    row_of = torch.zeros(T * topk, dtype=torch.int64, device=dev)
    row_w = torch.zeros(cap, dtype=torch.float32, device=dev)
    ws = torch.zeros(L.moe_dispatch_workspace_size(T, topk, E), dtype=torch.uint8, device=dev)
    L.moe_dispatch(torch.from_numpy(ids).to(dev), torch.from_numpy(w).to(dev), E, grp_off, grp_rows, row_src, row_of,
                   row_w, ws)
    assert L.device_status() == (ERR_ARG, WHERE_EXPERT_ID)
    flat = ids.reshape(-1)
    ok = (flat >= 0) & (flat < E)
    ro, rsrc, off = row_of.cpu().numpy(), row_src.cpu().numpy(), grp_off.cpu().numpy()
    assert np.all(ro[~ok] == -1)
    assert np.array_equal(grp_rows.cpu().numpy(), np.bincount(flat[ok], minlength=E))
    for p in np.nonzero(ok)[0]:
        r = ro[p]
        assert rsrc[r] == p and off[flat[p]] <= r < off[flat[p] + 1]
    # the same call on the in-range pairs' ids matches the oracle's stable order
    ids_ok = ids.copy()
    ids_ok[3, 1], ids_ok[10, 0] = 0, 0
    L.moe_dispatch(torch.from_numpy(ids_ok).to(dev), torch.from_numpy(w).to(dev), E, grp_off, grp_rows, row_src,
                   row_of, row_w, ws)
    assert L.device_status() == (0, 0)
    o_off, o_src = oracle.moe_dispatch(ids_ok, E)   # compact offsets; the GPU's groups start on 128-row blocks
    off, rows, rsrc = grp_off.cpu().numpy(), grp_rows.cpu().numpy(), row_src.cpu().numpy()
    assert np.array_equal(rows, np.diff(o_off))
    for g in range(E):
        assert np.array_equal(rsrc[off[g]:off[g] + rows[g]], o_src[o_off[g]:o_off[g + 1]])
