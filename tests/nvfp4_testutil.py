"""Test-side helpers: layout permutations between the oracle's logical layouts and the
library's blocked scale layout, operand upload, and the GEMM pass rule.  No quantization
arithmetic lives here."""
from __future__ import annotations

import numpy as np
import torch

# The GEMM pass rule.  The 2e-3 maximum relative error applies to the FP32-accumulated value;
# a bf16 output adds its own round-to-nearest step, at most half a bf16 ulp (up to 2^-8 of
# |y|, since bf16 carries 8 significant bits), which no bf16-output GEMM can avoid.  So
#   err_i = max(0, |y_i - ref_i| - halfulp_bf16(y_i)) / max(|ref_i|, rms(ref) / 64) <= 2e-3
# for bf16 outputs (halfulp = 0 for fp32 outputs), against the exact oracle product.  The
# rms/64 floor keeps outputs that cancel to nearly zero from turning an absolute error of
# fp32 size into a large relative one.
GEMM_RTOL = 2e-3


def sf_index(rows: int, ncols: int, sf_cols: int) -> np.ndarray:
    r = np.arange(rows, dtype=np.int64)[:, None]
    c = np.arange(ncols, dtype=np.int64)[None, :]
    return ((r >> 7) * (sf_cols >> 2) + (c >> 2)) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 + (c & 3)


def unswizzle(sf: torch.Tensor, rows: int, ncols: int, sf_cols: int, row0: int = 0) -> np.ndarray:
    """Blocked scale buffer -> logical [rows][ncols] scale bytes (rows row0 .. row0+rows)."""
    flat = sf.cpu().numpy()
    idx = sf_index(row0 + rows, ncols, sf_cols)[row0:]
    return flat[idx]


def swizzle_into(sf: torch.Tensor, logical: np.ndarray, sf_cols: int, row0: int = 0, col0: int = 0):
    rows, ncols = logical.shape
    idx = sf_index(row0 + rows, col0 + ncols, sf_cols)[row0:, col0:]
    flat = sf.cpu().numpy().copy()
    flat[idx] = logical
    sf.copy_(torch.from_numpy(flat))


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def tscale_fields(ts: torch.Tensor):
    t = ts.detach().cpu()
    f = t.numpy()
    e = t.view(torch.int32).numpy()
    return f[:, 0], f[:, 1], f[:, 2], e[:, 3]


def bf16_half_ulp(y: np.ndarray) -> np.ndarray:
    """Half the spacing of bf16 values around |y| (normal range): 2^(floor(log2|y|) - 8)."""
    a = np.abs(np.asarray(y, np.float64))
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a > 0, np.exp2(np.maximum(e, -126) - 8), 0.0)


def gemm_error(y: np.ndarray, ref: np.ndarray, out_bf16: bool = True) -> float:
    ref = np.asarray(ref, np.float64)
    y = np.asarray(y, np.float64)
    if not ref.size:
        return 0.0
    floor = np.sqrt(np.mean(ref * ref)) / 64
    den = np.maximum(np.abs(ref), floor)
    den[den == 0] = 1.0
    err = np.abs(y - ref)
    if out_bf16:
        err = np.maximum(err - bf16_half_ulp(y), 0.0)
    return float(np.max(err / den))


def normwise_error(y, ref) -> float:
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(np.asarray(y, np.float64) - ref)) / max(np.max(np.abs(ref)), 1e-300))
