"""Token-sharded activation quantization with Residual Activation Compensation, exact.

QUADS §3.3 scores each channel over the current token batch (Eq. (23)) and compensates the top k
of them (Eq. (24)); §4.1 runs the rollout engine with tensor parallelism.  When the rows (tokens)
of one batch are split over processes, every process reaches the unsplit batch's result exactly
with two small exchanges, because of what the batch-wide quantities are:

1. the FP32 tensor scale depends on the batch only through amax = max |x|.  Each process
   measures its own rows' amax (nvfp4_amax); a MAX all-reduce of one fp32 per group gives the
   batch's amax, and every process quantizes its rows with that same S_enc (nvfp4_quantize with
   the amax given);
2. a channel score is a sum over rows of exact integers.  The SUM all-reduce of the processes'
   partial scores (uint64 words carried as int64) is the batch's score bit for bit, whatever the
   order of summation;
3. the selection is a deterministic function of the scores, so every process selects the same
   channels (rac_select) and quantizes the residual of its own rows on them (rac_residual_tail).

The codes, block scales, selected channels and tail columns of every row then equal those of the
unsplit batch.  Exchanged per call: G x 4 fp32 and G x K int64 words per process (G row groups).

The row split itself is the caller's (each process holds its own rows); groups may be split
unevenly, and a process may hold no rows of a group.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import _lib as L
from .layers import Operand


class CudaShard:
    """One process's rows of a batch on its GPU: the activation operand (codes, blocked scales and
    tensor scales, with room for a k-column RAC tail), the channel scores and the selected
    channels, allocated once; every phase is one or two library calls on `stream`."""

    def __init__(self, rows: int, K: int, k: int, groups: int = 1, grp_off: Optional[torch.Tensor] = None,
                 grp_rows: Optional[torch.Tensor] = None, device="cuda", stream=None):
        self.rows, self.K, self.k, self.G = rows, K, k, groups
        self.grp_off, self.grp_rows = grp_off, grp_rows
        self.stream = stream
        self.a = Operand.empty(rows, K, k, groups, device=device)
        self.scores = torch.zeros(groups, K, dtype=torch.int64, device=device)
        self.idx = torch.zeros(groups, max(k, 1), dtype=torch.int32, device=device)

    def _groups(self):
        return dict(grp_off=self.grp_off, grp_rows=self.grp_rows, groups=self.G)

    def local_amax(self, x: torch.Tensor) -> torch.Tensor:
        """Phase 1: tensor scales [G, 4] fp32 with this process's amax in column 0 and zeros in the
        other columns (so that a MAX reduction of the whole tensor reduces the amax alone)."""
        L.nvfp4_amax(x, self.a.tscale, stream=self.stream, **self._groups())
        return self.a.tscale

    def quantize(self, x: torch.Tensor) -> torch.Tensor:
        """Phase 2 (after the amax reduction): codes and scales of this process's rows with the
        batch's tensor scale; returns this process's partial channel scores [G, K]."""
        L.nvfp4_quantize(x, self.a.codes, self.a.sf, self.a.sf_cols, self.a.tscale,
                         scores=self.scores if self.k else None, zero_pad=(self.k == 0), amax_given=True,
                         stream=self.stream, **self._groups())
        return self.scores

    def select_and_tail(self, x: torch.Tensor) -> None:
        """Phase 3 (after the score reduction): the batch's channel selection and this process's
        residual tail columns."""
        if self.k:
            L.rac_select_quantize(x, self.a.tscale, self.scores, self.k, self.a.codes, self.a.sf, self.a.sf_cols,
                                  self.idx, stream=self.stream, **self._groups())


def torch_all_reduce(group=None) -> Callable[[torch.Tensor, str], None]:
    """The exchanges through torch.distributed (NCCL for CUDA tensors, gloo for host tensors)."""
    import torch.distributed as dist

    ops = {"max": dist.ReduceOp.MAX, "sum": dist.ReduceOp.SUM}

    def reduce(t: torch.Tensor, op: str) -> None:
        dist.all_reduce(t, op=ops[op], group=group)

    return reduce


def rac_quantize_sharded(shard, x, all_reduce: Optional[Callable] = None):
    """Quantize + RAC of this process's rows `x` as part of the batch split over the processes of
    `all_reduce` (default: the default torch.distributed process group).

    `shard` provides the three phases (CudaShard on a GPU); the two exchanges between them are
    the only communication.  Every process must call this with its own rows, in the same order
    of calls.  Returns the shard, which holds the operand, the scores and the selection."""
    reduce = all_reduce if all_reduce is not None else torch_all_reduce()
    ts = shard.local_amax(x)
    reduce(ts, "max")      # amax >= 0 and the other columns are 0: the batch's amax per group
    if shard.k:
        scores = shard.quantize(x)
        reduce(scores, "sum")  # exact: integers, no overflow below 2^19 rows per group
    else:
        shard.quantize(x)
    shard.select_and_tail(x)
    return shard
