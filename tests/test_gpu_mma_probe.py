"""The NVFP4 MMA-rate probe (nvq_fp4_mma_rate), the roofline reference the bench reports beside
the GEMM: a short loop with and without the per-MMA scale copies returns a finite rate within
reach of the GPU's nominal dense NVFP4 peak, and leaves the device status clean."""
import math

import pytest
import torch

pytestmark = pytest.mark.gpu

NOMINAL_FP4_TFLOPS = 13500.0  # dense NVFP4, nominal, one GPU


@pytest.fixture(scope="module")
def L():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import _lib
    return _lib


@pytest.mark.parametrize("with_cp", [False, True])
def test_mma_rate_probe_runs_and_is_plausible(L, with_cp):
    tf = L.fp4_mma_rate(4096, with_cp=with_cp)
    assert math.isfinite(tf) and 0.05 * NOMINAL_FP4_TFLOPS < tf < 1.2 * NOMINAL_FP4_TFLOPS, tf
    assert L.device_status() == (0, 0)
