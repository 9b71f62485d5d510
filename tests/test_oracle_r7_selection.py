"""Reading R7 against the exact score on the workloads' token inputs.

QUADS §3.3 Eq. (23) scores channel j by the L2 norm of its residual over the token batch and
Eq. (24) keeps the top k.  The oracle (and the GPU) rank by the exact integer
score_j = sum_rows rint(|r| * 2^(20 - E))^2 instead, so that both sides pick identical channels
whatever the order of summation.  This test measures, on the actual inputs of the activation
workload (8192 x 4096), the dense GEMM workload (4096 x 4096) and the two MoE token batches,
how far the integer score is from the exact sum of squares (fp64, scaled by 2^(2(20 - E))), and
checks that the gap between the k-th and (k+1)-th exact sums exceeds twice that distance: the
integer top-k is then provably the exact-L2 top-k on these inputs, and the test also checks it
directly."""
import numpy as np
import pytest

import oracle
from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl


def _input(case: int):
    if case == 0:
        c = wl.CFG_ACT
        return c.name, c.make()[0], c.k
    if case == 1:
        c = wl.CFG_DENSE
        return c.name, wl.activations(c.M, c.K, c.seed, c.dist, c.x_scale, c.n_outliers, c.outlier_gain)[0], c.k
    c = (wl.CFG_MOE_PREFILL, wl.CFG_MOE_DECODE)[case - 2]
    return c.name + " (token input)", c.make_tokens()[0], c.k


@pytest.mark.slow
@pytest.mark.parametrize("case", list(range(4)), ids=["act_8192x4096", "dense_4096x4096", "moe_prefill_tokens",
                                                      "moe_decode_tokens"])
def test_integer_score_selects_the_exact_l2_top_k(case):
    name, x, k = _input(case)
    ts = oracle.tensor_scale(x)
    r = oracle.residual(x, ts).astype(np.float64)
    scale = 2.0 ** (2 * (20 - ts.shift_e))
    exact = (r * r).sum(axis=0) * scale          # sum of (|r| 2^(20-E))^2, exact enough in fp64
    score_u = oracle.scores(x, ts)
    score = score_u.astype(np.float64)
    dev = float(np.max(np.abs(score - exact)))    # rint moves each term by at most |r| s + 1/4
    srt = np.sort(exact)[::-1]
    gap = float(srt[k - 1] - srt[k])
    assert gap > 2 * dev, f"{name}: boundary gap {gap:.4g} not above twice the score deviation {dev:.4g}"
    order = np.lexsort((np.arange(exact.size), -exact))
    assert np.array_equal(oracle.topk(score_u, k), np.sort(order[:k])), name
