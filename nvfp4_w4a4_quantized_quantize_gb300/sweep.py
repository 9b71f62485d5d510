"""Residual channel ratio sweep (QUADS §4.3.3, Table 3): the compensated channel count k as a
share of the reduction width K, against the error it removes and the time it costs.

The paper reads the trade-off off the largest log-probability gap of whole RL runs at ratios of
12.5 % to 100 %.  Without a model, the same trade-off is measured here per layer, on the
synthetic workloads, with the layer's own kernels:

  act    X [8192, 4096], Student-t(3) x 0.5 with 1 % of the channels x20: the activation error
         of Eq. (21)'s compensated X~ (read back from the GEMM operand by rac_reconstruct),
         ||X~ - X||_F / ||X||_F and max |X~ - X|; the share of the outlier channels inside S;
         the time of quantize + select + residual tail.
  dense  Y = X W^T with M 4096, K 4096, N 14336: the output mismatch against the trainer's
         forward X W-hat^T (W4A16 of Eq. (12), W-hat = DQ(Q(W)) in fp32).  The weight mismatch
         is zero by construction (Eq. (16)), so this is the layer's activation share of the
         train/infer gap; also against X W^T (no weight quantization) for context; the forward
         time (quantize, select, residual and weight tails, GEMM).
  moe    the routed SwiGLU layer (16384 tokens, H 2048, 128 experts, top-8, I 768), k = ratio x H
         at gate/up and ratio x I at down: output mismatch against the fp32 layer on the same
         dequantized weights, and the step time (one CUDA-graph replay).

Ratio 0 is the layer without compensation.  k = ratio x K rounded down to a multiple of 16.
Error reductions are torch reductions over the kernels' outputs; the fp32 references are plain
torch fp32 matmuls with TF32 off.  Every time is the median of CUDA-graph replays, L2 flushed
before each.
"""
from __future__ import annotations

import contextlib

import numpy as np
import torch

from . import _lib as L
from . import workloads as wl
from .layers import MoERacLayer, Operand, RacLinear, quantize_weights
from .timing import time_graph_replays

RATIOS = (0.0, 0.125, 0.25, 0.5, 0.75, 1.0)


def k_of(ratio: float, K: int) -> int:
    return int(round(ratio * K)) // 16 * 16


def _bf16(bits: np.ndarray, dev) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(dev)


@contextlib.contextmanager
def _fp32_matmul():
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    try:
        yield
    finally:
        torch.backends.cuda.matmul.allow_tf32 = old


def _mismatch(y: torch.Tensor, ref: torch.Tensor) -> dict:
    d = y.float() - ref
    return {"rel_fro": float(d.norm() / ref.norm()), "rel_max": float(d.abs().max() / ref.abs().max())}


def _check_status():
    st, where = L.device_status()
    if st != 0:
        raise RuntimeError(f"device wait ran out ({where})")


def act_site(flush, steps, warmup, ratios=RATIOS, cfg=wl.CFG_ACT, dev="cuda") -> list:
    x_bits, _, outliers = cfg.make()
    M, K = cfg.M, cfg.K
    x = _bf16(x_bits, dev)
    xf = x.float()
    xnorm = float(xf.norm())
    recon = torch.empty(M, K, dtype=torch.float32, device=dev)
    rows = []
    for r in ratios:
        k = k_of(r, K)
        op = Operand.empty(M, K, k, 1, device=dev)
        scores = torch.zeros(K, dtype=torch.int64, device=dev)
        idx = torch.zeros(max(k, 1), dtype=torch.int32, device=dev)

        def fn():
            L.nvfp4_quantize(x, op.codes, op.sf, op.sf_cols, op.tscale, scores=scores if k else None,
                             zero_pad=(k == 0))
            if k:
                L.rac_select_quantize(x, op.tscale, scores, k, op.codes, op.sf, op.sf_cols, idx)

        ms = time_graph_replays(fn, flush, steps, warmup)
        fn()
        L.rac_reconstruct(op.codes, op.sf, op.sf_cols, op.tscale, K, k, idx if k else None, recon)
        torch.cuda.synchronize()
        _check_status()
        d = recon - xf
        sel = idx[:k].cpu().numpy()
        # algorithmic bytes: x read once per pass, codes + scales written, the tail likewise
        algo = M * K * (2 + 0.5 + 1 / 16) + M * k * (2 + 0.5 + 1 / 16)
        rows.append({"ratio": r, "k": k, "act_rel_fro": float(d.norm()) / xnorm, "act_max_abs": float(d.abs().max()),
                     "outlier_recall": float(np.isin(outliers, sel).mean()) if k else 0.0,
                     "ms": round(ms, 4), "gbs": round(algo / (ms * 1e-3) / 1e9, 1)})
        del op, scores, idx
    return rows


def dense_site(flush, steps, warmup, ratios=RATIOS, cfg=wl.CFG_DENSE, dev="cuda") -> list:
    x_bits, w_bits, _ = cfg.make()
    M, K, N = cfg.M, cfg.K, cfg.N
    x = _bf16(x_bits, dev)
    w = _bf16(w_bits, dev)
    w_hat = torch.empty(N, K, dtype=torch.float32, device=dev)
    quantize_weights(w, 0, w_hat=w_hat, w_hat_dtype=L.NVQ_F32)
    with _fp32_matmul():
        y_train = x.float() @ w_hat.t()
        y_full = x.float() @ w.float().t()
    del w_hat
    out = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    rows = []
    for r in ratios:
        k = k_of(r, K)
        lin = RacLinear(w, k, M)
        ms = time_graph_replays(lambda: lin.forward(x, out), flush, steps, warmup)
        lin.forward(x, out)
        torch.cuda.synchronize()
        _check_status()
        e_t, e_f = _mismatch(out, y_train), _mismatch(out, y_full)
        rows.append({"ratio": r, "k": k, "out_rel_fro_vs_w4a16": e_t["rel_fro"], "out_rel_max_vs_w4a16": e_t["rel_max"],
                     "out_rel_fro_vs_bf16": e_f["rel_fro"], "ms": round(ms, 4),
                     "useful_tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)})
        del lin
    return rows


def moe_reference_fp32(x: torch.Tensor, ids: torch.Tensor, tw: torch.Tensor, w13_hat: torch.Tensor,
                       w2_hat: torch.Tensor) -> torch.Tensor:
    """The routed SwiGLU layer in fp32: per expert, gate/up = x W13^T (gate the first I outputs),
    h = silu(gate) * up, y = h W2^T, summed over each token's experts with its routing weights."""
    T, H = x.shape
    I = w13_hat.shape[1] // 2
    out = torch.zeros(T, H, dtype=torch.float32, device=x.device)
    with _fp32_matmul():
        for e in range(w13_hat.shape[0]):
            tok, slot = (ids == e).nonzero(as_tuple=True)
            if tok.numel() == 0:
                continue
            gu = x[tok] @ w13_hat[e].t()
            g, u = gu[:, :I], gu[:, I:]
            h = g / (1.0 + torch.exp(-g)) * u
            out.index_add_(0, tok, (h @ w2_hat[e].t()) * tw[tok, slot].unsqueeze(1))
    return out


def moe_site(flush, steps, warmup, ratios=RATIOS, cfg=wl.CFG_MOE_PREFILL, dev="cuda") -> list:
    x_bits, ids, tw, outliers = cfg.make_tokens()
    w13_bits, w2_bits = cfg.make_weights()
    E, H, I, T, topk = cfg.E, cfg.H, cfg.I, cfg.T, cfg.topk
    w13 = _bf16(w13_bits.reshape(E * 2 * I, H), dev).view(E, 2 * I, H)
    w2 = _bf16(w2_bits.reshape(E * H, I), dev).view(E, H, I)
    del w13_bits, w2_bits
    x = _bf16(x_bits, dev)
    ids_d = torch.from_numpy(ids).to(dev)
    tw_d = torch.from_numpy(tw).to(dev)
    # dequantized weights exactly as the layer quantizes them (one tensor scale per expert)
    w13_hat = torch.empty(E, 2 * I, H, dtype=torch.float32, device=dev)
    w2_hat = torch.empty(E, H, I, dtype=torch.float32, device=dev)
    quantize_weights(w13, 0, w_hat=w13_hat, w_hat_dtype=L.NVQ_F32)
    quantize_weights(w2, 0, w_hat=w2_hat, w_hat_dtype=L.NVQ_F32)
    y_ref = moe_reference_fp32(x.float(), ids_d, tw_d, w13_hat, w2_hat)
    del w13_hat, w2_hat
    out = torch.empty(T, H, dtype=torch.bfloat16, device=dev)
    rows = []
    base_ms = None
    for r in ratios:
        k1, k2 = k_of(r, H), k_of(r, I)
        layer = MoERacLayer(w13, w2, k1, topk, T, k2=k2)
        ms = time_graph_replays(lambda: layer.forward(x, ids_d, tw_d, out), flush, steps, warmup)
        layer.forward(x, ids_d, tw_d, out)
        torch.cuda.synchronize()
        _check_status()
        base_ms = ms if base_ms is None else base_ms
        e = _mismatch(out, y_ref)
        sel = layer.idx1[:k1].cpu().numpy()
        rows.append({"ratio": r, "k_gate_up": k1, "k_down": k2, "out_rel_fro": e["rel_fro"], "out_rel_max": e["rel_max"],
                     "outlier_recall_tokens": float(np.isin(outliers, sel).mean()) if k1 else 0.0,
                     "ms": round(ms, 4), "tokens_per_s": round(T / (ms * 1e-3), 1),
                     "time_vs_ratio0": round(ms / base_ms, 4)})
        del layer
    return rows


def run(flush: torch.Tensor, steps: int, warmup: int, ratios=RATIOS) -> dict:
    return {"ratios": list(ratios), "act": act_site(flush, steps, warmup, ratios),
            "dense": dense_site(flush, steps, warmup, ratios), "moe": moe_site(flush, steps, warmup, ratios)}
