"""Test helpers: tolerance checks and readers of the library's device layouts.

The readers restate the layouts declared in include/hs.h in numpy, so that a
device result can be compared with the oracle's checkpoint-layout dequant."""
import numpy as np
import torch

import oracle

REL_L2 = 1e-3      # relative L2 error bound on fp32 outputs
MAX_ABS = 2e-3     # max-abs error bound, relative to max|y|


def check_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    scale = np.abs(ref).max()
    err = np.abs(got - ref)
    rel = np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300)
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e} > {REL_L2}"
    assert err.max() <= MAX_ABS * scale, f"{what}: max-abs {err.max():.3e} > {MAX_ABS}*{scale:.3e}"
    return rel, err.max() / max(scale, 1e-300)


def bf16_bits_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().float().numpy().astype(np.float64)


def check_bf16_within_one_ulp(y_bf16: torch.Tensor, ref: np.ndarray, what="", y_f32=None):
    """bf16 output contract.

    (a) if the kernel's fp32 sums are given, y_bf16 == RNE(y_f32) bit for bit;
    (b) y_bf16 equals RNE(ref) or a neighbour (one bf16 ulp) wherever |ref|
        exceeds the max-abs tolerance floor MAX_ABS * max|ref|; below that
        floor fp32 cancellation may exceed a bf16 ulp of the tiny value, and
        the bound is |y_bf16 - ref| <= MAX_ABS * max|ref| + ulp."""
    got = y_bf16.detach().cpu().view(torch.int16).numpy().astype(np.int64)
    if y_f32 is not None:
        own = torch.from_numpy(np.asarray(y_f32, dtype=np.float32)).to(torch.bfloat16)
        assert torch.equal(own.view(torch.int16), y_bf16.detach().cpu().view(torch.int16)), \
            f"{what}: bf16 output is not RNE of the kernel's fp32 sums"
    r = oracle.bf16_rne(ref)
    rb = torch.from_numpy(r.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().astype(np.int64)

    def ordered(b):  # bf16 bit patterns -> monotone integers
        b = b & 0xFFFF
        return np.where(b & 0x8000, -(b & 0x7FFF), b)

    d = np.abs(ordered(got) - ordered(rb))
    floor = MAX_ABS * np.abs(ref).max()
    big = np.abs(ref) > floor
    assert (d[big] <= 1).all(), f"{what}: bf16 differs from RNE(oracle) by {d[big].max()} ulp"
    yb = y_bf16.detach().cpu().float().numpy().astype(np.float64)
    small_err = np.abs(yb - ref)[~big]
    assert (small_err <= floor * 1.01 + 2.0 ** -133).all(), f"{what}: small outputs off by {small_err.max():.3e}"
    return int((d[big] == 1).sum())


def dequant_neuron_major(codes_nm: torch.Tensor, sb_nm: torch.Tensor) -> np.ndarray:
    """W[o][n] from the neuron-major layout: codes [N][H/2] (output 2j low nibble),
    sb [N/64][H] int32 = fp16 scale | fp16 bias << 16."""
    c = codes_nm.cpu().numpy()
    N, Hh = c.shape
    q = np.empty((N, 2 * Hh), dtype=np.float64)
    q[:, 0::2] = c & 15
    q[:, 1::2] = c >> 4
    sb = sb_nm.cpu().numpy().view(np.uint32)
    s = (sb & 0xFFFF).astype(np.uint16).view(np.float16).astype(np.float64)
    b = (sb >> 16).astype(np.uint16).view(np.float16).astype(np.float64)
    s = np.repeat(s, 64, axis=0)
    b = np.repeat(b, 64, axis=0)
    return (s * q + b).T


def live_flip_bound(x, up, n_rows=None) -> np.ndarray:
    """Per neuron, the largest |z| whose sign fp32 accumulation may flip:
    gamma * sum_k |w_nk x_k| with gamma = K * 2^-24 (K = hidden)."""
    w = oracle.dequant(up)
    xa = np.abs(oracle.as_f64(x))
    return (w.shape[1] * 2.0 ** -24) * (np.abs(w) @ xa)


def check_bf16_rounding(y_bf16: torch.Tensor, y_f32, ref: np.ndarray, what=""):
    """bf16 output contract when the arithmetic itself uses 16-bit operands
    (prefill): y_bf16 == RNE(y_f32) bit for bit, and every element within the
    max-abs bar of the oracle plus half a bf16 ulp (the final rounding).
    Returns the largest distance in bf16 ulps from RNE(ref)."""
    own = torch.from_numpy(np.asarray(y_f32, dtype=np.float32)).to(torch.bfloat16)
    assert torch.equal(own.view(torch.int16), y_bf16.detach().cpu().view(torch.int16)), \
        f"{what}: bf16 output is not RNE of the kernel's fp32 sums"
    ref = np.asarray(ref, dtype=np.float64)
    yb = y_bf16.detach().cpu().float().numpy().astype(np.float64)
    _, e = np.frexp(np.where(ref != 0, ref, 1.0))
    half_ulp = np.ldexp(1.0, np.maximum(e - 1, -126) - 8)
    bound = MAX_ABS * np.abs(ref).max() + half_ulp * 1.001
    err = np.abs(yb - ref)
    assert (err <= bound).all(), f"{what}: bf16 error {err.max():.3e} above the bar"
    return float((np.abs(yb - oracle.bf16_rne(ref)) / (2 * half_ulp)).max())
