"""Re-quantisation of a down projection with its scales along the neuron axis
(test infrastructure: fp32 decisions restated plainly, fp64 dequantisation).

"Skipping dead neurons..." (sevren.ai), section "The whole decode step": the
checkpoint keeps one scale per group of 64 neurons, laid along the output
axis, so a single live neuron costs its group's scales; re-quantising with the
scales along the neuron axis would remove that toll (the page measured a small
perplexity cost and kept the checkpoint bytes).

Reading (the page gives no method): for each neuron n and each group j of 64
consecutive outputs, min-max affine 4-bit quantisation of the checkpoint's
dequantised weights w[o][n], o = 64j .. 64j+63:
    scale = fp16((max - min) / 15),  bias = fp16(min),
    q     = clamp(rint((w - bias) / scale), 0, 15)   (q = 0 where scale = 0).
The integer decisions are taken in fp32, the precision the GPU kernel uses:
w is the exact dequantised value rounded once to fp32, and each step above
rounds to fp32 (IEEE, round to nearest even); fp16 conversions round to
nearest even.  Dequantisation w' = scale * q + bias is then exact in fp64.
"""
from __future__ import annotations

import numpy as np

from .moe import dequant, unpack_codes

__all__ = ["requant_down_rowscale", "dequant_rowscale"]


def requant_down_rowscale(down):
    """Checkpoint-layout down projection [H][N] -> (codes uint8 [N][H/2], output
    2j in the low nibble of byte j; scale fp16 [N][H/64]; bias fp16 [N][H/64])."""
    W = dequant(down)                       # exact, fp64 [H][N]
    H, N = W.shape
    w = W.astype(np.float32).T.reshape(N, H // 64, 64)   # [n][j][k] = w[64j + k][n]
    mx, mn = w.max(axis=2), w.min(axis=2)
    s16 = ((mx - mn) / np.float32(15)).astype(np.float16)
    b16 = mn.astype(np.float16)
    sf = s16.astype(np.float32)[..., None]
    bf = b16.astype(np.float32)[..., None]
    with np.errstate(divide="ignore", invalid="ignore"):
        qf = np.rint((w - bf) / sf)
    q = np.where(sf == 0, np.float32(0), np.clip(qf, 0, 15)).astype(np.uint8).reshape(N, H)
    codes = (q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8)
    return codes, s16, b16


def dequant_rowscale(codes, scale, bias) -> np.ndarray:
    """fp64 matrix [H][N] of a row-scale down projection (the layout above)."""
    q = unpack_codes(codes).astype(np.float64)            # [N][H]
    s = np.repeat(np.asarray(scale, dtype=np.float64), 64, axis=-1)
    b = np.repeat(np.asarray(bias, dtype=np.float64), 64, axis=-1)
    return (s * q + b).T
