"""Seeded synthetic inputs for the NVFP4 W4A4 + RAC rollout path.

This module only draws random numbers and rounds them to bf16 storage; it holds none of the
quantizer's, the selection's or the GEMM's arithmetic.  Both the CUDA path (tests, bench) and
the CPU oracle consume the bytes it returns.

The paper's workload (MoE 25B-A2.8B rollout on competition-math and code prompts, QUADS §4.1)
needs model weights and datasets that are not available, so these generators stand in for it:
Gaussian or Student-t activations with a few outlier channels that imitate the persistent
vertical residual bands of QUADS Fig. 4(a), Gaussian weights, and top-8 MoE routing.

All draws use numpy's PCG64 with an explicit seed; fp64 (or fp32 for the large weight tensors)
values are rounded to nearest-even bf16 and returned as their uint16 bit patterns.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


def to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float values to bf16 (nearest, ties to even) and return the uint16 bit patterns."""
    f = np.ascontiguousarray(a, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (h.astype(np.uint32) << 16).view(np.float32)


def _normal_f32(rng: np.random.Generator, shape, std: float, chunk: int = 1 << 24) -> np.ndarray:
    n = int(np.prod(shape))
    out = np.empty(n, np.uint16)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        v = rng.standard_normal(e - s, dtype=np.float32)
        v *= np.float32(std)
        out[s:e] = to_bf16_bits(v)
    return out.reshape(shape)


def activations(M: int, K: int, seed: int, dist: str = "normal", scale: float = 1.0,
                n_outliers: int = 0, outlier_gain: float = 1.0):
    """X [M, K] bf16 bits and the sorted outlier channel list.

    dist "normal": N(0, 1); "student_t3": Student-t with 3 degrees of freedom.  The whole matrix
    is multiplied by ``scale``; ``n_outliers`` channels, drawn without replacement by the same
    generator, are multiplied by ``outlier_gain`` (in fp64, before the bf16 rounding).
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    if dist == "normal":
        x = rng.standard_normal((M, K))
    elif dist == "student_t3":
        x = rng.standard_t(3.0, (M, K))
    else:
        raise ValueError(dist)
    x *= scale
    ch = np.sort(rng.choice(K, size=n_outliers, replace=False)) if n_outliers else np.zeros(0, np.int64)
    if n_outliers:
        x[:, ch] *= outlier_gain
    return to_bf16_bits(x), ch


def weights(shape, std: float, seed: int) -> np.ndarray:
    """W ~ N(0, std^2) in bf16 bits (fp32 draws, chunked so that large tensors stay cheap)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    return _normal_f32(rng, shape, std)


def routing_zipf(T: int, E: int, topk: int, s: float, seed: int):
    """Top-k routing from softmax(N(0,1) logits + b_e), b_e = log p_e, p_e ~ rank_e^-s over a
    seeded permutation of the experts.  Returns ids [T, topk] int32 (descending probability)
    and the renormalised top-k probabilities [T, topk] float32."""
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(E)
    p = np.empty(E)
    p[perm] = np.arange(1, E + 1, dtype=np.float64) ** (-s)
    p /= p.sum()
    logits = rng.standard_normal((T, E)) + np.log(p)[None, :]
    return _topk_softmax(logits, topk)


def routing_uniform(T: int, E: int, topk: int, seed: int):
    """Uniform-random routing: each token picks ``topk`` distinct experts uniformly; its gate
    weights are the renormalised softmax of N(0,1) logits on those experts."""
    rng = np.random.Generator(np.random.PCG64(seed))
    keys = rng.random((T, E))
    ids = np.argsort(keys, axis=1)[:, :topk].astype(np.int32)
    logits = rng.standard_normal((T, topk))
    w = np.exp(logits - logits.max(axis=1, keepdims=True))
    w /= w.sum(axis=1, keepdims=True)
    return ids, w.astype(np.float32)


def _topk_softmax(logits: np.ndarray, topk: int):
    z = np.exp(logits - logits.max(axis=1, keepdims=True))
    prob = z / z.sum(axis=1, keepdims=True)
    ids = np.argsort(-prob, axis=1, kind="stable")[:, :topk].astype(np.int32)
    w = np.take_along_axis(prob, ids, axis=1)
    w /= w.sum(axis=1, keepdims=True)
    return ids, w.astype(np.float32)


# ------------------------------------------------------------------------- the five workloads
@dataclass(frozen=True)
class DenseLinear:
    """One RAC linear layer: X [M, K] @ W [N, K]^T with k compensated channels."""
    name: str
    M: int
    K: int
    N: int
    k: int
    seed: int
    dist: str = "normal"
    x_scale: float = 1.0
    n_outliers: int = 0
    outlier_gain: float = 1.0
    w_std: float = 0.02

    def make(self):
        x, ch = activations(self.M, self.K, self.seed, self.dist, self.x_scale, self.n_outliers,
                            self.outlier_gain)
        w = weights((self.N, self.K), self.w_std, self.seed + 1) if self.N else None
        return x, w, ch


@dataclass(frozen=True)
class MoELayer:
    """Routed SwiGLU expert layer: gate/up GEMM (N = 2I), SwiGLU, down GEMM (K = I), combine."""
    name: str
    T: int
    H: int
    E: int
    topk: int
    I: int
    k: int
    seed: int
    routing: str = "zipf"
    zipf_s: float = 1.1
    n_outliers: int = 0
    outlier_gain: float = 20.0
    w_std: float = 0.02

    def make_tokens(self):
        x, ch = activations(self.T, self.H, self.seed, "normal", 1.0, self.n_outliers, self.outlier_gain)
        if self.routing == "zipf":
            ids, w = routing_zipf(self.T, self.E, self.topk, self.zipf_s, self.seed + 7)
        else:
            ids, w = routing_uniform(self.T, self.E, self.topk, self.seed + 7)
        return x, ids, w, ch

    def make_weights(self):
        w13 = weights((self.E, 2 * self.I, self.H), self.w_std, self.seed + 11)
        w2 = weights((self.E, self.H, self.I), self.w_std, self.seed + 13)
        return w13, w2


# Small single linear layer; the oracle finishes it in well under a second.
CFG_SMALL = DenseLinear("linear_64x256x256_k16", M=64, K=256, N=256, k=16, seed=0,
                        n_outliers=4, outlier_gain=16.0)
# Activation quantizer + RAC only (HBM-bound): Student-t(3) * 0.5 with 1 % outlier channels x20.
CFG_ACT = DenseLinear("actquant_rac_8192x4096_k64", M=8192, K=4096, N=0, k=64, seed=1,
                      dist="student_t3", x_scale=0.5, n_outliers=41, outlier_gain=20.0)
# Dense prefill-shaped W4A4 + RAC GEMM.
CFG_DENSE = DenseLinear("dense_rac_gemm_4096x4096x14336_k64", M=4096, K=4096, N=14336, k=64,
                        seed=2, n_outliers=41, outlier_gain=20.0)
# MoE expert layer, prefill/rollout batch, Zipf(1.1)-skewed routing.
CFG_MOE_PREFILL = MoELayer("moe_prefill_T16384_H2048_E128_top8_I768_k32", T=16384, H=2048, E=128,
                           topk=8, I=768, k=32, seed=3, routing="zipf", n_outliers=20)
# Decode-shaped MoE step (uniform routing); also the trainer-side weight QDQ of all experts.
CFG_MOE_DECODE = MoELayer("moe_decode_T512_H4096_E128_top8_I1536_k64", T=512, H=4096, E=128,
                          topk=8, I=1536, k=64, seed=4, routing="uniform", n_outliers=41)

ALL = [CFG_SMALL, CFG_ACT, CFG_DENSE, CFG_MOE_PREFILL, CFG_MOE_DECODE]
