"""GPU parity of the tcgen05 block-scaled W4A4 + RAC (grouped) GEMM against the exact oracle.

Operands are built by the oracle (so this file isolates the GEMM), uploaded in the library's
blocked scale layout, and the GEMM call rebuilds the weight tail itself; the tail must equal
the oracle's bit for bit and the output must pass the 2e-3 rule against the exact product."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import GEMM_RTOL, gemm_error, swizzle_into, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 31)
    return _lib


def _ts_tensor(tss):
    arr = np.zeros((len(tss), 4), np.float32)
    for i, t in enumerate(tss):
        arr[i, :3] = [t.amax, t.s_enc, t.s_dec]
        arr[i, 3:4] = np.array([t.shift_e], np.int32).view(np.float32)
    return torch.from_numpy(arr).cuda()


class Op:
    def __init__(self, L, rows, ktot):
        self.ld = max(16, (ktot // 2 + 15) // 16 * 16)
        self.sf_cols = L.sf_cols(ktot)
        self.codes = torch.zeros(rows, self.ld, dtype=torch.uint8, device="cuda")
        self.sf = torch.zeros(L.sf_bytes(rows, self.sf_cols), dtype=torch.uint8, device="cuda")

    def put(self, row0, codes, scales, col0=0):
        c = self.codes.cpu().numpy()
        c[row0:row0 + codes.shape[0], col0 // 2:col0 // 2 + codes.shape[1]] = codes
        self.codes.copy_(torch.from_numpy(c))
        swizzle_into(self.sf, scales, self.sf_cols, row0=row0, col0=col0 // 16)


def _run_case(L, counts, N, K, k, epilogue=0, seed=0, dense=False, rows_extra=0, out_amax=False):
    """counts: rows per group.  Groups start on multiples of 128 unless dense (one group)."""
    G = len(counts)
    off = [0]
    for c in counts:
        off.append(off[-1] + (c if dense else (c + 127) // 128 * 128))
    rows = max(off[-1] + rows_extra, 1)
    ktot = K + k
    A = Op(L, rows, ktot)
    B = Op(L, G * N, ktot)
    rng = np.random.default_rng(seed)
    a_ts, b_ts, a_full, b_full, idxs = [], [], [], [], []
    for g, c in enumerate(counts):
        x, _ = wl.activations(max(c, 1), K, seed=seed * 100 + g, n_outliers=max(1, K // 64), outlier_gain=12.0)
        x = x[:c] if c else x[:0]
        w = wl.weights((N, K), 0.02, seed=seed * 100 + 50 + g)
        wts = oracle.tensor_scale(w)
        wc, ws = oracle.quantize(w, wts)
        B.put(g * N, wc, ws)
        b_ts.append(wts)
        if c:
            q = oracle.rac_quantize(x, k)
            A.put(off[g], np.concatenate([q.codes, q.tail_codes], 1), np.concatenate([q.scales, q.tail_scales], 1))
            a_ts.append(q.ts)
            idx = q.idx
        else:
            a_ts.append(oracle.tensor_scale_from_amax(1.0))
            idx = np.sort(rng.choice(K, k, replace=False)).astype(np.int32)
        idxs.append(idx)
        if k:
            tc, tsc = oracle.weight_tail(wc, ws, wts, idx)
            b_full.append((np.concatenate([wc, tc], 1), np.concatenate([ws, tsc], 1)))
        else:
            b_full.append((wc, ws))
        a_full.append(q if c else None)
    idx_t = torch.from_numpy(np.stack(idxs) if k else np.zeros((G, 1), np.int32)).cuda()
    out_w = N // 2 if epilogue == 1 else N
    out = torch.full((rows, out_w), float("nan"), dtype=torch.float32 if epilogue == 3 else torch.bfloat16,
                     device="cuda")
    row_w = torch.from_numpy(rng.uniform(0.1, 1.0, rows).astype(np.float32)).cuda()
    out_ts = torch.full((G, 4), 7.0, dtype=torch.float32, device="cuda") if out_amax else None
    go = torch.tensor(off, dtype=torch.int64, device="cuda")
    gr = torch.tensor(counts, dtype=torch.int64, device="cuda")
    L.w4a4_rac_grouped_gemm(A.codes, A.sf, A.sf_cols, _ts_tensor(a_ts), B.codes, B.sf, B.sf_cols, _ts_tensor(b_ts),
                            N, K, k, idx_t if k else None, out, groups=G, grp_off=None if dense else go,
                            grp_rows=None if dense else gr, rows=rows, a_scale_per_group=True,
                            idx_per_group=True, epilogue=epilogue, row_w=row_w if epilogue == 2 else None,
                            out_tscale=out_ts)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0), "a device-side wait ran out"
    # the weight tail the call built
    bc = B.codes.cpu().numpy()
    bsl = unswizzle(B.sf, G * N, B.sf_cols, B.sf_cols)
    y = out.float().cpu().numpy()
    worst = 0.0
    for g, c in enumerate(counts):
        wfc, wfs = b_full[g]
        assert np.array_equal(bc[g * N:(g + 1) * N, :ktot // 2], wfc), f"weight tail of group {g}"
        assert np.array_equal(bsl[g * N:(g + 1) * N, :ktot // 16], wfs)
        assert not bsl[g * N:(g + 1) * N, ktot // 16:].any()
        if not c:
            continue
        q = a_full[g]
        ac = np.concatenate([q.codes, q.tail_codes], 1)
        asc = np.concatenate([q.scales, q.tail_scales], 1)
        ref = oracle.gemm(ac, asc, wfc, wfs, q.ts.s_dec, b_ts[g].s_dec)
        if epilogue == 1:
            I = N // 2
            ref = oracle.swiglu(ref[:, :I], ref[:, I:]).reshape(c, I)
        elif epilogue == 2:
            ref = ref * row_w[off[g]:off[g] + c].cpu().numpy()[:, None].astype(np.float64)
        got = y[off[g]:off[g] + c]
        assert np.all(np.isfinite(got))
        if out_amax:
            # the epilogue's per-group amax is the max |stored bf16| over the group's rows, exactly
            ots = out_ts.cpu().numpy()
            assert ots[g, 0] == np.float32(np.abs(got).max()), (g, ots[g, 0], np.abs(got).max())
        worst = max(worst, gemm_error(got, ref, out_bf16=(epilogue != 3)))
    if out_amax:
        ots = out_ts.cpu().numpy()
        for g, c in enumerate(counts):
            if not c:
                assert ots[g, 0] == 0.0
        assert not ots[:, 1:].any()  # the rest of each record is zeroed
    # rows outside every group are not written
    if not dense:
        valid = np.zeros(rows, bool)
        for g, c in enumerate(counts):
            valid[off[g]:off[g] + c] = True
        assert np.all(np.isnan(y[~valid]))
    assert worst <= GEMM_RTOL, worst
    return worst


def test_gemm_small_linear_layer(L):
    """The small linear layer: M=64, K=256, N=256, k=16."""
    _run_case(L, [64], 256, 256, 16, dense=True)


@pytest.mark.parametrize("M,N,K,k", [(1, 256, 256, 0), (200, 512, 448, 64), (130, 256, 320, 16),
                                     (256, 512, 4096, 64), (77, 768, 1536, 48),
                                     (130, 256, 256, 256), (200, 512, 1024, 512)])
def test_gemm_dense_shapes(L, M, N, K, k):
    _run_case(L, [M], N, K, k, dense=True, seed=M + K)


def test_gemm_grouped_store(L):
    _run_case(L, [0, 130, 7, 256, 1], 256, 512, 32, seed=3)


def test_gemm_grouped_swiglu(L):
    _run_case(L, [129, 0, 40], 512, 768, 32, epilogue=1, seed=4)


def test_gemm_grouped_row_scale(L):
    _run_case(L, [33, 300], 256, 768, 64, epilogue=2, seed=5)


def test_gemm_fp32_output_is_elementwise_within_2e3(L):
    """The FP32-accumulated product itself, stored without the bf16 rounding: the strict
    elementwise rule (no rounding allowance)."""
    worst = _run_case(L, [200, 3, 128], 512, 1536, 64, epilogue=3, seed=6)
    assert worst < 1e-5


@pytest.mark.parametrize("epilogue", [1, 2])
def test_gemm_epilogue_amax_for_the_next_quantizer(L, epilogue):
    """out_tscale: zeroed, then per group max |out| over the rows the call stores (bit-exact),
    with an empty group left at 0 -- what nvfp4_quantize(amax_given) takes as the amax."""
    _run_case(L, [300, 0, 129, 1], 512, 256, 32, epilogue=epilogue, seed=7, out_amax=True)
