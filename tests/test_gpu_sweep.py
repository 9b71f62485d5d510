"""The residual channel ratio sweep on small workloads: it runs through the layer's kernels, and
the activation error it reports falls as the ratio grows (the channel sets are nested and the
second pass never increases an element's error)."""
import pytest
import torch

from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

RATIOS = (0.0, 0.125, 0.5, 1.0)


@pytest.fixture(scope="module")
def env():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from nvfp4_w4a4_quantized_quantize_gb300 import sweep
    return sweep, torch.empty(1 << 20, dtype=torch.uint8, device="cuda")


def test_sweep_act_site_error_falls_with_k(env):
    sweep, flush = env
    cfg = wl.DenseLinear("act_small", M=300, K=512, N=0, k=0, seed=9, dist="student_t3", x_scale=0.5,
                         n_outliers=5, outlier_gain=20.0)
    rows = sweep.act_site(flush, 2, 1, RATIOS, cfg=cfg)
    errs = [r["act_rel_fro"] for r in rows]
    assert [r["k"] for r in rows] == [0, 64, 256, 512]
    assert all(a >= b for a, b in zip(errs, errs[1:])) and errs[-1] < 0.5 * errs[0], errs
    assert rows[1]["outlier_recall"] == 1.0  # 5 outlier channels x20 are all among the top 64


def test_sweep_dense_and_moe_sites_run(env):
    sweep, flush = env
    dense = wl.DenseLinear("dense_small", M=256, K=512, N=512, k=0, seed=10, n_outliers=5, outlier_gain=20.0)
    rows = sweep.dense_site(flush, 2, 1, RATIOS, cfg=dense)
    e = [r["out_rel_fro_vs_w4a16"] for r in rows]
    assert e[-1] < e[0], e
    moe = wl.MoELayer("moe_small", T=256, H=256, E=8, topk=2, I=128, k=0, seed=11, n_outliers=3)
    rows = sweep.moe_site(flush, 2, 1, RATIOS, cfg=moe)
    assert [(r["k_gate_up"], r["k_down"]) for r in rows] == [(0, 0), (32, 16), (128, 64), (256, 128)]
    e = [r["out_rel_fro"] for r in rows]
    assert e[-1] < e[0], e
