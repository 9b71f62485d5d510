"""The bounded-wait path of the quantizer's copy ring, run for real.

Every shared-memory wait of quant_score_kernel is bounded by nvq_set_wait_limit.  With a limit of
a few cycles, waits for stages still in flight from HBM run out: the kernel records
NVQ_ERR_TIMEOUT in the device status word, lets the copies it already issued land (under a bound
of its own, which the configurable limit does not shrink) and returns.  The test checks that the
status reaches the host through nvq_device_status, that the context stays usable, and that the
next call at the default limit is bit-exact against the oracle again.  No wait is left unbounded
and no copy outlives its CTA, so the GPU is never hung or faulted."""
import numpy as np
import pytest
import torch

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
from tests.nvfp4_testutil import bf16_tensor, unswizzle

pytestmark = pytest.mark.gpu

DEFAULT_LIMIT = 1 << 32
QUANT_WAIT_SITES = {21, 22, 23}  # loader slot wait, loader drain, compute stage wait


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    yield _lib
    _lib.set_wait_limit(DEFAULT_LIMIT)


def test_quantizer_wait_times_out_and_recovers(L):
    M, K = 16384, 4096  # 128 MB of bf16: the ring's stages arrive from HBM, far beyond a few cycles
    x_bits, _ = wl.activations(M, K, seed=77, n_outliers=41, outlier_gain=20.0)
    x = bf16_tensor(x_bits)
    sfc = L.sf_cols(K)
    codes = torch.zeros(M, K // 2, dtype=torch.uint8, device="cuda")
    sf = torch.zeros(L.sf_bytes(M, sfc), dtype=torch.uint8, device="cuda")
    ts = torch.zeros(1, 4, dtype=torch.float32, device="cuda")
    scores = torch.zeros(K, dtype=torch.int64, device="cuda")
    flush = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
    assert L.device_status() == (0, 0)

    timed_out = None
    try:
        for limit in (1, 4, 16):
            flush.zero_()
            L.set_wait_limit(limit)
            L.nvfp4_quantize(x, codes, sf, sfc, ts, scores=scores, zero_pad=True)
            torch.cuda.synchronize()  # the kernel returned: the context is usable
            st, where = L.device_status()
            if st != 0:
                timed_out = (st, where)
                break
    finally:
        L.set_wait_limit(DEFAULT_LIMIT)
    assert timed_out is not None, "no wait ran out at a limit of a few cycles"
    assert timed_out[0] == 5 and timed_out[1] in QUANT_WAIT_SITES, timed_out  # NVQ_ERR_TIMEOUT
    assert L.device_status() == (0, 0), "reading the status clears it"

    # the same call at the default limit is exact again
    codes.fill_(0xAB)
    L.nvfp4_quantize(x, codes, sf, sfc, ts, scores=scores, zero_pad=True)
    torch.cuda.synchronize()
    assert L.device_status() == (0, 0)
    rows = np.r_[0:64, M // 2:M // 2 + 64, M - 64:M]
    t = oracle.tensor_scale(x_bits)
    oc, os_ = oracle.quantize(np.ascontiguousarray(x_bits[rows]), t)
    assert np.array_equal(codes.cpu().numpy()[rows], oc)
    assert np.array_equal(unswizzle(sf, M, K // 16, sfc)[rows], os_)
    assert np.array_equal(scores.cpu().numpy().view(np.uint64), oracle.scores(x_bits, t))
