"""Trainer-side W4A16 QAT node (QUADS §3.2, Eq. (12)-(13)): the learner's W-hat equals the
rollout's dequantized weight bit for bit (Eq. (15)-(16): zero weight mismatch), the forward is
x W-hat^T, and the backward is the straight-through estimator."""
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
    return _lib


def test_qat_weight_is_the_rollout_dequantized_weight(L):
    from nvfp4_w4a4_quantized_quantize_gb300.layers import RacLinear
    from nvfp4_w4a4_quantized_quantize_gb300.qat import qdq_weight
    N, K = 384, 272
    w_bits = wl.weights((N, K), 0.02, seed=71)
    w = bf16_tensor(w_bits)
    w_hat = qdq_weight(w)
    # the oracle's DQ(Q(W)), rounded to bf16
    t = oracle.tensor_scale(w_bits)
    oc, os_ = oracle.quantize(w_bits, t)
    ref = oracle.bf16_round(oracle.dequantize(oc, os_, t.s_dec))
    assert np.array_equal(w_hat.cpu().view(torch.int16).numpy().view(np.uint16), ref)
    # the rollout layer's stored operand, dequantized on the host: the same values (Eq. (16))
    lin = RacLinear(w, 16, 128)
    torch.cuda.synchronize()
    codes = lin.w.codes.cpu().numpy()[:, :K // 2]
    scales = unswizzle(lin.w.sf, N, K // 16, lin.w.sf_cols)
    s_dec = lin.w.tscale.cpu().numpy()[0, 2]
    assert s_dec == np.float32(t.s_dec)
    assert np.array_equal(oracle.bf16_round(oracle.dequantize(codes, scales, s_dec)), ref)


def test_qat_forward_and_straight_through_backward(L):
    from nvfp4_w4a4_quantized_quantize_gb300.qat import QATLinear, qdq_weight
    torch.manual_seed(3)
    lin = QATLinear(512, 256)
    x = torch.randn(4, 64, 512, device="cuda").bfloat16().requires_grad_(True)
    y = lin(x)
    gy = torch.randn_like(y)
    y.backward(gy)
    w_hat = qdq_weight(lin.weight)
    # reference: a plain linear layer whose weight is W-hat, differentiated by autograd
    x2 = x.detach().clone().requires_grad_(True)
    w2 = w_hat.detach().clone().requires_grad_(True)
    y2 = x2 @ w2.t()
    y2.backward(gy)
    assert torch.equal(y, y2)
    assert torch.equal(x.grad, x2.grad)                 # dL/dx = dL/dy W-hat
    assert torch.equal(lin.weight.grad, w2.grad)        # STE: dL/dW = dL/dW-hat
    # the weight is discretized (it differs from the master copy) but the gradient is not masked
    assert not torch.equal(w_hat, lin.weight.detach())


def test_qat_grouped_expert_weights(L):
    from nvfp4_w4a4_quantized_quantize_gb300.qat import qdq_weight
    G, N, K = 3, 128, 256
    w_bits = wl.weights((G, N, K), 0.02, seed=72)
    w_hat = qdq_weight(bf16_tensor(w_bits.reshape(G * N, K)).view(G, N, K))
    for g in range(G):
        t = oracle.tensor_scale(w_bits[g])
        oc, os_ = oracle.quantize(w_bits[g], t)
        ref = oracle.bf16_round(oracle.dequantize(oc, os_, t.s_dec))
        assert np.array_equal(w_hat[g].cpu().view(torch.int16).numpy().view(np.uint16), ref)
