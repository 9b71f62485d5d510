"""The token-sharded quantize + RAC path (rows of one batch split over processes), on CPU with
gloo and two ranks.  Each rank runs the oracle's steps on its own rows through the product's
driver `rac_quantize_sharded`, which all-reduces the amax (MAX) and the integer channel scores
(SUM) between the phases.  The selected channels, codes, block scales and residual tails must
equal the oracle's `rac_quantize` on the whole batch bit for bit (QUADS §3.3 Eq. (23)-(24): the
score and the selection are over the current token batch)."""
import multiprocessing as mp
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
K, k, SPLIT, M = 256, 32, 50, 97


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _batch():
    sys.path.insert(0, ROOT)
    from nvfp4_w4a4_quantized_quantize_gb300 import workloads as wl
    # outlier channels in one half only, so that each half alone would select differently
    x, _ = wl.activations(M, K, seed=21, n_outliers=6, outlier_gain=12.0)
    x2, _ = wl.activations(M, K, seed=22, n_outliers=6, outlier_gain=12.0)
    x[SPLIT:] = x2[SPLIT:]
    return x


class OracleShard:
    """The three phases of a shard done by the oracle on host arrays (bf16 bit patterns)."""

    def __init__(self, k_):
        self.k = k_

    def local_amax(self, x):
        import oracle
        import torch
        self.ts_t = torch.tensor([[oracle.tensor_scale(x).amax, 0.0, 0.0, 0.0]], dtype=torch.float32)
        return self.ts_t

    def quantize(self, x):
        import oracle
        import torch
        self.ts = oracle.tensor_scale_from_amax(float(self.ts_t[0, 0]))
        self.codes, self.scales = oracle.quantize(x, self.ts)
        self.scores = torch.from_numpy(oracle.scores(x, self.ts).view(np.int64).copy()).reshape(1, -1)
        return self.scores

    def select_and_tail(self, x):
        import oracle
        s = self.scores.numpy().reshape(-1).view(np.uint64)
        self.idx = oracle.topk(s, self.k)
        self.tail_codes, self.tail_scales = oracle.rac_tail(x, self.ts, self.idx)


def _worker(rank, port, q):
    try:
        sys.path.insert(0, ROOT)
        os.environ.update(WORLD_SIZE="2", RANK=str(rank), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        import torch.distributed as dist
        from nvfp4_w4a4_quantized_quantize_gb300.sharded import rac_quantize_sharded
        dist.init_process_group(backend="gloo")
        x = _batch()
        rows = slice(0, SPLIT) if rank == 0 else slice(SPLIT, M)
        sh = rac_quantize_sharded(OracleShard(k), np.ascontiguousarray(x[rows]))
        dist.destroy_process_group()
        q.put((rank, sh.ts.amax, sh.ts.s_enc, sh.ts.s_dec, sh.ts.shift_e, sh.codes, sh.scales, sh.idx,
               sh.tail_codes, sh.tail_scales, sh.scores.numpy().view(np.uint64)))
    except Exception as e:  # report instead of hanging the parent
        q.put(("error", repr(e)))


def test_two_rank_token_sharded_rac_equals_whole_batch():
    import oracle
    port = _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=180) for _ in range(2)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert all(r[0] != "error" for r in res), res
    res.sort(key=lambda r: r[0])
    x = _batch()
    full = oracle.rac_quantize(x, k)
    for r in res:
        assert (r[1], r[2], r[3], r[4]) == (full.ts.amax, full.ts.s_enc, full.ts.s_dec, full.ts.shift_e)
        assert np.array_equal(r[7], full.idx)
        assert np.array_equal(r[10].reshape(-1), full.scores)
    for name, i, part in (("codes", 5, full.codes), ("scales", 6, full.scales), ("tail codes", 8, full.tail_codes),
                          ("tail scales", 9, full.tail_scales)):
        assert np.array_equal(np.concatenate([res[0][i], res[1][i]]), part), name
    # the exchanges matter: either half alone selects another channel set
    for rows in (slice(0, SPLIT), slice(SPLIT, M)):
        assert not np.array_equal(oracle.rac_quantize(np.ascontiguousarray(x[rows]), k).idx, full.idx)


def test_sharded_driver_reduces_amax_then_scores():
    """The driver's order of phases and exchanges, with a recording reduction (one process)."""
    sys.path.insert(0, ROOT)
    import torch
    from nvfp4_w4a4_quantized_quantize_gb300.sharded import rac_quantize_sharded
    log = []

    class Fake:
        k = 16

        def local_amax(self, x):
            log.append("amax")
            return torch.zeros(1, 4)

        def quantize(self, x):
            log.append("quantize")
            return torch.zeros(1, 8, dtype=torch.int64)

        def select_and_tail(self, x):
            log.append("select")

    def reduce(t, op):
        log.append(f"reduce-{op}-{t.dtype}")

    rac_quantize_sharded(Fake(), None, all_reduce=reduce)
    assert log == ["amax", "reduce-max-torch.float32", "quantize", "reduce-sum-torch.int64", "select"]
    Fake.k = 0
    log.clear()
    rac_quantize_sharded(Fake(), None, all_reduce=reduce)
    assert log == ["amax", "reduce-max-torch.float32", "quantize", "select"]
