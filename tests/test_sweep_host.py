"""Host logic of the residual channel ratio sweep, on the CPU: the ratio -> k rounding, and the
fp32 MoE reference the sweep measures the layer against (checked token by token against the
layer's definition: gate rows first in W13, SwiGLU, down projection, routing-weighted sum)."""
import numpy as np
import torch

from nvfp4_w4a4_quantized_quantize_gb300 import sweep


def test_k_of_rounds_down_to_tail_blocks():
    assert [sweep.k_of(r, 2048) for r in sweep.RATIOS] == [0, 256, 512, 1024, 1536, 2048]
    assert [sweep.k_of(r, 768) for r in sweep.RATIOS] == [0, 96, 192, 384, 576, 768]
    assert sweep.k_of(0.125, 100) == 0 and sweep.k_of(0.5, 100) == 48


def test_moe_reference_fp32_token_by_token():
    rng = np.random.default_rng(5)
    T, H, E, I, topk = 9, 32, 4, 16, 2
    x = rng.standard_normal((T, H)).astype(np.float32)
    w13 = (rng.standard_normal((E, 2 * I, H)) * 0.1).astype(np.float32)
    w2 = (rng.standard_normal((E, H, I)) * 0.1).astype(np.float32)
    ids = np.stack([rng.choice(E, topk, replace=False) for _ in range(T)]).astype(np.int64)
    tw = rng.uniform(0.1, 1.0, (T, topk)).astype(np.float32)
    got = sweep.moe_reference_fp32(torch.from_numpy(x), torch.from_numpy(ids), torch.from_numpy(tw),
                                   torch.from_numpy(w13), torch.from_numpy(w2)).numpy()
    ref = np.zeros((T, H))
    for t in range(T):
        for s in range(topk):
            e = ids[t, s]
            gu = w13[e].astype(np.float64) @ x[t].astype(np.float64)
            g, u = gu[:I], gu[I:]
            h = g / (1.0 + np.exp(-g)) * u
            ref[t] += tw[t, s] * (w2[e].astype(np.float64) @ h)
    assert np.allclose(got, ref, rtol=1e-5, atol=1e-6)
