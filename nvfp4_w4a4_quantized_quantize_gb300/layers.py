"""The rollout-side RAC linear layer and MoE expert layer, composed from the C-ABI calls.

Every arithmetic step runs in libnvfp4rac.so; this module only allocates buffers once (torch
device memory) and issues the calls on one stream, so a forward pass makes no allocation and
can be captured in a CUDA graph.

QUADS (arXiv 2607.15810) §3.3: activations are quantized online (Eq. (9)), the k channels with
the largest residual norm are selected per forward pass (Eq. (23)-(24)), their residual is
quantized a second time and carried as extra K-columns of the same W4A4 GEMM (Eq. (21)).
§3.2: weights are quantized once by the same quantizer the trainer's QDQ uses (Eq. (12)).
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import torch

from . import _lib as L


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclass
class Operand:
    """An NVFP4 GEMM operand: codes [rows, ld] (two per byte), blocked UE4M3 scales, tensor scales."""
    codes: torch.Tensor
    sf: torch.Tensor
    sf_cols: int
    tscale: torch.Tensor  # float32 [G, 4]: amax, s_enc, s_dec, shift_e (int32 bits)
    rows: int
    K: int
    k: int

    @staticmethod
    def empty(rows: int, K: int, k_max: int, groups: int = 1, device="cuda") -> "Operand":
        ktot = K + k_max
        # rows start on 128-byte boundaries: a GEMM K-stage reads a 128-byte slice of each row,
        # which then lies in one L2 line instead of two (K + k columns are rarely a multiple of
        # 256); TMA fills of such slices from DRAM ran 1.9x faster, from L2 1.1x
        ld = _round_up(max(ktot // 2, 16), 128)
        cols = L.sf_cols(ktot)
        codes = torch.zeros(rows, ld, dtype=torch.uint8, device=device)
        sf = torch.zeros(L.sf_bytes(rows, cols), dtype=torch.uint8, device=device)
        ts = torch.zeros(groups, 4, dtype=torch.float32, device=device)
        return Operand(codes, sf, cols, ts, rows, K, k_max)


@dataclass
class ChannelMajor:
    """Channel-major copy of a quantized weight operand (nvfp4_channel_major), read by the
    weight tail: codes [G, K, N/2] (rows 2m, 2m+1 of a channel in one byte), scales [G, K/16, N]."""
    codes: torch.Tensor
    sf: torch.Tensor

    @staticmethod
    def of(op: Operand, G: int, N: int, stream=None) -> Optional["ChannelMajor"]:
        if N % 64:
            return None
        K = op.K
        cm = ChannelMajor(torch.empty(G, K, N // 2, dtype=torch.uint8, device=op.codes.device),
                          torch.empty(G, K // 16, N, dtype=torch.uint8, device=op.codes.device))
        L.nvfp4_channel_major(G, N, K, op.codes, op.sf, op.sf_cols, cm.codes, cm.sf, stream=stream)
        return cm


def quantize_weights(w: torch.Tensor, k_max: int, w_hat: Optional[torch.Tensor] = None,
                     w_hat_dtype: int = L.NVQ_BF16) -> Operand:
    """W [G, N, K] (or [N, K]) bf16 -> NVFP4 operand with room for a k_max-column RAC tail."""
    w3 = w if w.dim() == 3 else w.unsqueeze(0)
    G, N, K = w3.shape
    op = Operand.empty(G * N, K, k_max, G, device=w.device)
    L.weight_qdq(w3, G, N, K, op.codes, op.sf, op.sf_cols, op.tscale, w_hat=w_hat, w_hat_dtype=w_hat_dtype)
    return op


def _weight_tail(op: Operand, cm: Optional[ChannelMajor], G: int, N: int, k: int, idx: torch.Tensor,
                 idx_per_group: bool = False, stream=None):
    L.rac_weight_tail(G, N, op.K, k, idx, op.codes, op.sf, op.sf_cols, op.tscale, idx_per_group=idx_per_group,
                      cm_codes=cm.codes if cm else None, cm_sf=cm.sf if cm else None, stream=stream)


class RacLinear:
    """Dense rollout linear layer Y = X W^T with NVFP4 W4A4 + RAC (k compensated channels)."""

    def __init__(self, w: torch.Tensor, k: int, max_rows: int):
        self.N, self.K = w.shape
        self.k = k
        self.w = quantize_weights(w, k)
        self.w_cm = ChannelMajor.of(self.w, 1, self.N) if k else None
        self.a = Operand.empty(max_rows, self.K, k, 1, device=w.device)
        self.scores = torch.zeros(self.K, dtype=torch.int64, device=w.device)
        self.idx = torch.zeros(max(k, 1), dtype=torch.int32, device=w.device)

    def forward(self, x: torch.Tensor, out: torch.Tensor, k: Optional[int] = None, stream=None):
        k = self.k if k is None else k
        M = x.shape[0]
        L.nvfp4_quantize(x, self.a.codes, self.a.sf, self.a.sf_cols, self.a.tscale,
                         scores=self.scores if k else None, zero_pad=(k == 0), stream=stream)
        if k:
            L.rac_select_quantize(x, self.a.tscale, self.scores, k, self.a.codes, self.a.sf, self.a.sf_cols,
                                  self.idx, stream=stream)
            _weight_tail(self.w, self.w_cm, 1, self.N, k, self.idx, stream=stream)
        L.w4a4_rac_grouped_gemm(self.a.codes, self.a.sf, self.a.sf_cols, self.a.tscale, self.w.codes, self.w.sf,
                                self.w.sf_cols, self.w.tscale, self.N, self.K, k, None, out,
                                rows=M, stream=stream)
        return out


# Stages of MoERacLayer.forward that its `events` argument can time, in launch order.
MOE_STAGES = ("dispatch", "quant_rac_tokens", "weight_tail_w13", "gather", "gemm_gate_up", "quant_h", "select_h",
              "weight_tail_w2", "tail_h", "gemm_down", "combine")


class MoERacLayer:
    """Routed SwiGLU expert layer with NVFP4 W4A4 + RAC in both expert GEMMs.

    gate/up:  A = Q(X) per token with one channel set S over all tokens (the W13 site of QUADS
              §3.3), gathered into the routed layout; fused gate/up weights W13 [E, 2I, H];
              SwiGLU in the GEMM epilogue -> h [routed rows, I] bf16.
    down:     h quantized with one tensor scale and one channel set per expert; W2 [E, H, I];
              the routing weight is applied in the GEMM epilogue -> y; combine sums the topk
              rows of every token.
    """

    def __init__(self, w13: torch.Tensor, w2: torch.Tensor, k: int, topk: int, max_tokens: int,
                 k2: Optional[int] = None, side_stream: bool = True):
        """k: compensated channels at the gate/up site (of H), k2 at the down site (of I; default k).
        side_stream: run the work that does not depend on dispatch (token quantization and
        selection, the weight tails) on a second stream; False issues everything in order on the
        caller's stream."""
        dev = w13.device
        self.E, twoI, self.H = w13.shape
        self.I = twoI // 2
        k2 = k if k2 is None else k2
        self.k, self.k2, self.topk, self.T = k, k2, topk, max_tokens
        self.w13 = quantize_weights(w13, k)
        self.w2 = quantize_weights(w2, k2)
        self.w13_cm = ChannelMajor.of(self.w13, self.E, twoI) if k else None
        self.w2_cm = ChannelMajor.of(self.w2, self.E, self.H) if k2 else None
        cap = L.moe_capacity(max_tokens, topk, self.E)
        self.cap = cap
        E = self.E
        self.grp_off = torch.zeros(E + 1, dtype=torch.int64, device=dev)
        self.grp_rows = torch.zeros(E, dtype=torch.int64, device=dev)
        self.row_src = torch.zeros(cap, dtype=torch.int32, device=dev)
        self.row_of = torch.zeros(max_tokens * topk, dtype=torch.int64, device=dev)
        self.row_w = torch.zeros(cap, dtype=torch.float32, device=dev)
        self.ws = torch.zeros(L.moe_dispatch_workspace_size(max_tokens, topk, E), dtype=torch.uint8, device=dev)
        self.a_tok = Operand.empty(max_tokens, self.H, k, 1, device=dev)
        self.scores1 = torch.zeros(self.H, dtype=torch.int64, device=dev)
        self.idx1 = torch.zeros(max(k, 1), dtype=torch.int32, device=dev)
        self.a_routed = Operand.empty(cap, self.H, k, 1, device=dev)
        self.h = torch.zeros(cap, self.I, dtype=torch.bfloat16, device=dev)
        self.a2 = Operand.empty(cap, self.I, k2, E, device=dev)
        self.scores2 = torch.zeros(E, self.I, dtype=torch.int64, device=dev)
        self.idx2 = torch.zeros(E, max(k2, 1), dtype=torch.int32, device=dev)
        self.y = torch.zeros(cap, self.H, dtype=torch.bfloat16, device=dev)
        # side stream for the work that does not depend on dispatch (token quantization and
        # selection) or on the gather (the gate/up weight tail); events fork and join it, so
        # a CUDA graph captured around forward() holds the two branches in parallel
        self.side = torch.cuda.Stream(device=dev) if side_stream else None
        self.ev_fork = torch.cuda.Event()
        self.ev_tok = torch.cuda.Event()
        self.ev_wt = torch.cuda.Event()
        self.ev_sel2 = torch.cuda.Event()
        self.ev_wt2 = torch.cuda.Event()

    def kernel_launches_per_step(self) -> int:
        """Kernels one forward() launches: dispatch 4; tokens: amax + quantize 2, selection and
        residual tail 2; gather 1; gate/up: weight tail 1, GEMM 1; h: quantize 1 (its amax comes
        from the GEMM epilogue), selection and residual tail 2; down: weight tail 1, GEMM 1;
        combine 1.  A site without RAC (k = 0) has no selection, residual or weight tail."""
        rac1 = 1 if self.k else 0
        rac2 = 1 if self.k2 else 0
        tok = 2 + 2 * rac1
        h = 1 + 2 * rac2
        return 4 + tok + 1 + (rac1 + 1) + h + (rac2 + 1) + 1

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, out: torch.Tensor,
                stream=None, events: Optional[dict] = None):
        """events: optional dict that receives (start, end) CUDA events around each stage (for
        per-kernel timing): 'dispatch', 'quant_rac_tokens', 'weight_tail_w13', 'gather',
        'gemm_gate_up', 'quant_h', 'select_h', 'weight_tail_w2', 'tail_h', 'gemm_down' and
        'combine' (stages a site without RAC does not run are absent)."""
        T = x.shape[0]
        k, k2, E, H, I = self.k, self.k2, self.E, self.H, self.I
        st = torch.cuda.current_stream() if stream is None else stream
        side = self.side if self.side is not None else st

        def mark(name, pos, on=None):
            if events is not None:
                ev = events.setdefault(name, (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                ev[pos].record(st if on is None else on)

        # fork: token quantization + selection on the side stream, dispatch on the main one
        self.ev_fork.record(st)
        side.wait_event(self.ev_fork)
        mark("quant_rac_tokens", 0, side)
        L.nvfp4_quantize(x, self.a_tok.codes, self.a_tok.sf, self.a_tok.sf_cols, self.a_tok.tscale,
                         scores=self.scores1 if k else None, zero_pad=(k == 0), stream=side)
        if k:
            L.rac_select_quantize(x, self.a_tok.tscale, self.scores1, k, self.a_tok.codes, self.a_tok.sf,
                                  self.a_tok.sf_cols, self.idx1, stream=side)
        mark("quant_rac_tokens", 1, side)
        self.ev_tok.record(side)
        mark("dispatch", 0)
        L.moe_dispatch(topk_ids, topk_w, E, self.grp_off, self.grp_rows, self.row_src, self.row_of, self.row_w,
                       self.ws, stream=st)
        mark("dispatch", 1)
        st.wait_event(self.ev_tok)
        # the gate/up weight tail (needs the selection only) beside the gather
        if k:
            mark("weight_tail_w13", 0, side)
            _weight_tail(self.w13, self.w13_cm, E, 2 * I, k, self.idx1, stream=side)
            mark("weight_tail_w13", 1, side)
        self.ev_wt.record(side)
        mark("gather", 0)
        L.nvfp4_gather_rows(self.a_tok.codes, self.a_tok.sf, self.a_tok.sf_cols, T, self.row_src, self.topk, H + k,
                            self.a_routed.codes, self.a_routed.sf, stream=st)
        mark("gather", 1)
        st.wait_event(self.ev_wt)  # join
        mark("gemm_gate_up", 0)
        L.w4a4_rac_grouped_gemm(self.a_routed.codes, self.a_routed.sf, self.a_routed.sf_cols, self.a_tok.tscale,
                                self.w13.codes, self.w13.sf, self.w13.sf_cols, self.w13.tscale, 2 * I, H, k,
                                None, self.h, groups=E, grp_off=self.grp_off, grp_rows=self.grp_rows,
                                rows=self.cap, epilogue=L.NVQ_EPI_SWIGLU, out_tscale=self.a2.tscale, stream=st)
        mark("gemm_gate_up", 1)
        # down input: per-expert tensor scale (amax of h measured by the gate/up epilogue) and
        # channel set
        mark("quant_h", 0)
        L.nvfp4_quantize(self.h, self.a2.codes, self.a2.sf, self.a2.sf_cols, self.a2.tscale,
                         scores=self.scores2 if k2 else None, grp_off=self.grp_off, grp_rows=self.grp_rows,
                         groups=E, zero_pad=(k2 == 0), amax_given=True, stream=st)
        mark("quant_h", 1)
        if k2:
            # selection, then the down weight tail (needs idx2 only) beside the residual tail of h
            mark("select_h", 0)
            L.rac_select(self.scores2, I, k2, self.idx2, groups=E, stream=st)
            mark("select_h", 1)
            self.ev_sel2.record(st)
            side.wait_event(self.ev_sel2)
            mark("weight_tail_w2", 0, side)
            _weight_tail(self.w2, self.w2_cm, E, H, k2, self.idx2, idx_per_group=True, stream=side)
            mark("weight_tail_w2", 1, side)
            self.ev_wt2.record(side)
            mark("tail_h", 0)
            L.rac_residual_tail(self.h, self.a2.tscale, self.idx2, k2, self.a2.codes, self.a2.sf, self.a2.sf_cols,
                                grp_off=self.grp_off, grp_rows=self.grp_rows, groups=E, stream=st)
            mark("tail_h", 1)
            st.wait_event(self.ev_wt2)
        mark("gemm_down", 0)
        L.w4a4_rac_grouped_gemm(self.a2.codes, self.a2.sf, self.a2.sf_cols, self.a2.tscale, self.w2.codes,
                                self.w2.sf, self.w2.sf_cols, self.w2.tscale, H, I, k2, None,
                                self.y, groups=E, grp_off=self.grp_off, grp_rows=self.grp_rows, rows=self.cap,
                                a_scale_per_group=True, idx_per_group=True, epilogue=L.NVQ_EPI_ROW_SCALE,
                                row_w=self.row_w, stream=st)
        mark("gemm_down", 1)
        mark("combine", 0)
        L.moe_combine(self.y, self.row_of, T, self.topk, H, out, stream=st)
        mark("combine", 1)
        return out


@dataclass
class Fp8Operand:
    """An FP8 GEMM operand: E4M3 codes [rows, ld] and blocked UE8M0 tile scales."""
    codes: torch.Tensor
    sf: torch.Tensor
    sf_cols: int

    @staticmethod
    def empty(rows: int, K: int, device="cuda") -> "Fp8Operand":
        cols = L.fp8_sf_cols(K)
        return Fp8Operand(torch.zeros(rows, _round_up(K, 16), dtype=torch.uint8, device=device),
                          torch.zeros(L.sf_bytes(rows, cols), dtype=torch.uint8, device=device), cols)


class Fp8MoELayer:
    """The same routed SwiGLU expert layer as MoERacLayer on the FP8 W8A8 baseline the paper
    compares against (§2.2 "FP8", §4.4.2): E4M3 activations with a power-of-two scale per
    1 x 128 tile, E4M3 weights with one per 128 x 128 tile, block-scaled tcgen05 GEMMs.

    dispatch; tokens -> FP8 (fp8_quantize); gather into the routed layout; gate/up GEMM with the
    SwiGLU epilogue -> h; h -> FP8 (every routed row, padding rows included: they hold zeros);
    down GEMM with the routing-weight epilogue -> y; combine."""

    def __init__(self, w13: torch.Tensor, w2: torch.Tensor, topk: int, max_tokens: int):
        dev = w13.device
        self.E, twoI, self.H = w13.shape
        self.I = twoI // 2
        self.topk, self.T = topk, max_tokens
        E, H, I = self.E, self.H, self.I
        self.w13 = Fp8Operand.empty(E * twoI, H, device=dev)
        L.fp8_quantize(w13.reshape(E * twoI, H), self.w13.codes, self.w13.sf, self.w13.sf_cols, tile_rows=128)
        self.w2 = Fp8Operand.empty(E * H, I, device=dev)
        L.fp8_quantize(w2.reshape(E * H, I), self.w2.codes, self.w2.sf, self.w2.sf_cols, tile_rows=128)
        cap = L.moe_capacity(max_tokens, topk, E)
        self.cap = cap
        self.grp_off = torch.zeros(E + 1, dtype=torch.int64, device=dev)
        self.grp_rows = torch.zeros(E, dtype=torch.int64, device=dev)
        self.row_src = torch.zeros(cap, dtype=torch.int32, device=dev)
        self.row_of = torch.zeros(max_tokens * topk, dtype=torch.int64, device=dev)
        self.row_w = torch.zeros(cap, dtype=torch.float32, device=dev)
        self.ws = torch.zeros(L.moe_dispatch_workspace_size(max_tokens, topk, E), dtype=torch.uint8, device=dev)
        self.a_tok = Fp8Operand.empty(max_tokens, H, device=dev)
        self.a_routed = Fp8Operand.empty(cap, H, device=dev)
        self.h = torch.zeros(cap, I, dtype=torch.bfloat16, device=dev)
        self.a2 = Fp8Operand.empty(cap, I, device=dev)
        self.y = torch.zeros(cap, H, dtype=torch.bfloat16, device=dev)

    def kernel_launches_per_step(self) -> int:
        """dispatch 4, token quantize 1, gather 1, gate/up GEMM 1, h quantize 1, down GEMM 1, combine 1."""
        return 10

    def forward(self, x: torch.Tensor, topk_ids: torch.Tensor, topk_w: torch.Tensor, out: torch.Tensor, stream=None):
        T = x.shape[0]
        E, H, I = self.E, self.H, self.I
        L.moe_dispatch(topk_ids, topk_w, E, self.grp_off, self.grp_rows, self.row_src, self.row_of, self.row_w,
                       self.ws, stream=stream)
        L.fp8_quantize(x, self.a_tok.codes, self.a_tok.sf, self.a_tok.sf_cols, tile_rows=1, stream=stream)
        L.fp8_gather_rows(self.a_tok.codes, self.a_tok.sf, self.a_tok.sf_cols, T, self.row_src, self.topk, H,
                          self.a_routed.codes, self.a_routed.sf, stream=stream)
        L.fp8_blockscaled_grouped_gemm(self.a_routed.codes, self.a_routed.sf, self.a_routed.sf_cols, self.w13.codes,
                                       self.w13.sf, self.w13.sf_cols, 2 * I, H, self.h, groups=E, grp_off=self.grp_off,
                                       grp_rows=self.grp_rows, rows=self.cap, epilogue=L.NVQ_EPI_SWIGLU, stream=stream)
        L.fp8_quantize(self.h, self.a2.codes, self.a2.sf, self.a2.sf_cols, tile_rows=1, stream=stream)
        L.fp8_blockscaled_grouped_gemm(self.a2.codes, self.a2.sf, self.a2.sf_cols, self.w2.codes, self.w2.sf,
                                       self.w2.sf_cols, H, I, self.y, groups=E, grp_off=self.grp_off,
                                       grp_rows=self.grp_rows, rows=self.cap, epilogue=L.NVQ_EPI_ROW_SCALE,
                                       row_w=self.row_w, stream=stream)
        L.moe_combine(self.y, self.row_of, T, self.topk, H, out, stream=stream)
        return out
