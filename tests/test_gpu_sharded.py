"""The token-sharded quantize + RAC path on one GPU: the rows of one batch split into two shards
(CudaShard), with the two exchanges of rac_quantize_sharded done in-process (MAX of the tensor
scales, SUM of the integer scores) since this run has one GPU.  Every shard's codes, scales,
selection and tail columns must equal the unsplit batch's, which the quantizer tests check
against the oracle; the dense case is compared with the oracle directly as well."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import bf16_tensor, unswizzle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    _lib.set_wait_limit(1 << 31)
    return _lib


def _two_shards(shards, xs):
    """rac_quantize_sharded's phases for two shards in one process, with the two reductions."""
    ts = [s.local_amax(x) for s, x in zip(shards, xs)]
    m = torch.maximum(ts[0], ts[1])
    for s in shards:
        s.a.tscale.copy_(m)
    sc = [s.quantize(x).clone() for s, x in zip(shards, xs)]
    tot = sc[0] + sc[1]
    for s in shards:
        s.scores.copy_(tot)
    for s, x in zip(shards, xs):
        s.select_and_tail(x)
    torch.cuda.synchronize()


def _unsplit(L, x, k, groups=1, grp_off=None):
    from nvfp4_w4a4_quantized_quantize_gb300.layers import Operand
    a = Operand.empty(x.shape[0], x.shape[1], k, groups)
    sc = torch.zeros(groups, x.shape[1], dtype=torch.int64, device="cuda")
    idx = torch.zeros(groups, k, dtype=torch.int32, device="cuda")
    L.nvfp4_quantize(x, a.codes, a.sf, a.sf_cols, a.tscale, scores=sc, grp_off=grp_off, groups=groups)
    L.rac_select_quantize(x, a.tscale, sc, k, a.codes, a.sf, a.sf_cols, idx, grp_off=grp_off, groups=groups)
    torch.cuda.synchronize()
    return a, sc, idx


def _same_rows(a_full, rows_full, a_sh, rows_sh, K, k):
    assert torch.equal(a_full.codes[rows_full], a_sh.codes[rows_sh])
    n_full, n_sh = a_full.codes.shape[0], a_sh.codes.shape[0]
    f = unswizzle(a_full.sf, n_full, (K + k) // 16, a_full.sf_cols)[rows_full.cpu().numpy()]
    s = unswizzle(a_sh.sf, n_sh, (K + k) // 16, a_sh.sf_cols)[rows_sh.cpu().numpy()]
    assert np.array_equal(f, s)


def test_two_shards_equal_the_unsplit_batch_dense(L):
    from nvfp4_w4a4_quantized_quantize_gb300.sharded import CudaShard
    M, K, k, cut = 1000, 2048, 64, 333
    x_bits, _ = wl.activations(M, K, seed=41, n_outliers=20, outlier_gain=20.0)
    x = bf16_tensor(x_bits)
    xs = [x[:cut].contiguous(), x[cut:].contiguous()]
    shards = [CudaShard(cut, K, k), CudaShard(M - cut, K, k)]
    _two_shards(shards, xs)
    assert L.device_status() == (0, 0)
    a, sc, idx = _unsplit(L, x, k)
    for s, rows in zip(shards, (torch.arange(0, cut, device="cuda"), torch.arange(cut, M, device="cuda"))):
        assert torch.equal(s.a.tscale, a.tscale)
        assert torch.equal(s.scores, sc)
        assert torch.equal(s.idx, idx)
        _same_rows(a, rows, s.a, torch.arange(rows.numel(), device="cuda"), K, k)
    q = oracle.rac_quantize(x_bits, k)
    assert np.array_equal(idx.cpu().numpy()[0], q.idx)
    assert np.array_equal(a.codes.cpu().numpy()[:, :K // 2], q.codes)
    assert np.array_equal(a.codes.cpu().numpy()[:, K // 2:(K + k) // 2], q.tail_codes)


def test_two_shards_equal_the_unsplit_batch_grouped(L):
    """Row groups (per-expert tensor scales and selections, the down projection's input), each
    group split unevenly between the shards; one shard holds no row of the last group."""
    from nvfp4_w4a4_quantized_quantize_gb300.sharded import CudaShard
    K, k = 768, 32
    sizes = [300, 129, 64, 5]
    cuts = [100, 129, 1, 5]  # rows of each group on shard 0 (group 3 wholly on shard 0)
    M = sum(sizes)
    x_bits, _ = wl.activations(M, K, seed=43, n_outliers=8, outlier_gain=20.0)
    x = bf16_tensor(x_bits)
    off = np.concatenate([[0], np.cumsum(sizes)])
    rows0 = np.concatenate([np.arange(off[g], off[g] + cuts[g]) for g in range(4)])
    rows1 = np.concatenate([np.arange(off[g] + cuts[g], off[g + 1]) for g in range(4)])
    off0 = np.concatenate([[0], np.cumsum(cuts)])
    off1 = np.concatenate([[0], np.cumsum(np.array(sizes) - np.array(cuts))])
    G = 4
    dev = "cuda"
    r0, r1 = torch.from_numpy(rows0).to(dev), torch.from_numpy(rows1).to(dev)
    xs = [x[r0].contiguous(), x[r1].contiguous()]
    shards = [CudaShard(len(rows0), K, k, G, grp_off=torch.from_numpy(off0).to(dev)),
              CudaShard(len(rows1), K, k, G, grp_off=torch.from_numpy(off1).to(dev))]
    _two_shards(shards, xs)
    assert L.device_status() == (0, 0)
    a, sc, idx = _unsplit(L, x, k, G, torch.from_numpy(off).to(dev))
    for s, rows in zip(shards, (r0, r1)):
        assert torch.equal(s.a.tscale, a.tscale)
        assert torch.equal(s.scores, sc)
        assert torch.equal(s.idx, idx)
        _same_rows(a, rows, s.a, torch.arange(rows.numel(), device=dev), K, k)
