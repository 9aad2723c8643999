"""Seeded synthetic inputs: checkpoint-layout W4 experts, activations, logits.

Shapes follow the workloads described on "Skipping dead neurons: a faster
Nemotron 3.5 Lightning on Apple silicon" (sections "Inside a MoE layer" and
"Two projections and a switch"): hidden size 2688, routed experts of 1856
neurons, a shared expert of 3712 neurons, 128 routed experts, top-6 routing,
4-bit affine weights with one fp16 scale and bias per group of 64 inputs.

Storage of a projection W of shape [rows][cols] (row = output of the
projection, col = input; groups of 64 run along the input axis), the
"checkpoint layout":
  codes  uint8 [rows][cols/2]   code of column 2j in the low nibble of byte j,
                                code of column 2j+1 in the high nibble
  scale  fp16  [rows][cols/64]
  bias   fp16  [rows][cols/64]
For the up projection rows are neurons and cols the hidden axis; for the
down projection rows are the hidden outputs and cols the neurons.

Random numbers.  Bulk weight bytes and scales come from a counter-based
integer hash evaluated with torch integer ops, so that the same tensor is
produced bit for bit on the CPU and on a GPU, and so that any single expert
can be regenerated without generating the others (its values depend only on
the stream key and the element index).  Normal draws (activations, logits,
single-expert pre-activations) come from numpy's PCG64 seeded per stream.

Calibration of the live fraction.  Each neuron gets a pre-activation offset
off_n = Phi^-1(p) * ||w_n||_2 so that, for x ~ N(0, I), P(w_n . x + off_n > 0)
equals p.  Because this generator always stores bias = -8 * scale, the
dequantised up row is w_{n,k} = scale_{n,g}*(q_{n,k} - 8) and its squared norm
is sum_g scale_{n,g}^2 * sum_{k in g} (q_{n,k} - 8)^2, evaluated from exact
integer group sums and fp64 scale squares in a fixed order.  Permanently dead
neurons get off_n = -inf.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass

import numpy as np
import torch
from scipy.special import ndtri

__all__ = [
    "HIDDEN", "N_ROUTED", "N_SHARED", "N_EXPERTS", "TOP_K", "GROUP",
    "stream_key", "hash_u32", "random_code_bytes", "random_scales",
    "W4Proj", "Expert", "gen_proj", "gen_expert", "gen_routed_stack", "stack_offsets",
    "code_group_sq_sums", "calibrated_offsets", "dead_mask",
    "normal_f32", "normal_bf16", "expert_down_h", "shared_live_fraction",
    "uniform_f64",
]

HIDDEN = 2688
N_ROUTED = 1856
N_SHARED = 3712
N_EXPERTS = 128
TOP_K = 6
GROUP = 64

_M32 = 0xFFFFFFFF
# odd multipliers below 2^31 so that x * c with x < 2^32 stays below 2^63
_C1 = 0x21F0AAAD
_C2 = 0x735A2D97


def stream_key(*parts) -> tuple[int, int]:
    """Two 32-bit keys for a named random stream (seed, config, layer, ...)."""
    d = hashlib.blake2b(repr(tuple(parts)).encode(), digest_size=8).digest()
    return int.from_bytes(d[:4], "little"), int.from_bytes(d[4:], "little")


def _seed_ints(*parts) -> list[int]:
    d = hashlib.blake2b(repr(tuple(parts)).encode(), digest_size=16).digest()
    return [int.from_bytes(d[i:i + 4], "little") for i in range(0, 16, 4)]


def _mix32(x: torch.Tensor) -> torch.Tensor:
    # xorshift-multiply rounds on values held in int64, kept below 2^32
    x = x ^ (x >> 16)
    x = (x * _C1) & _M32
    x = x ^ (x >> 15)
    x = (x * _C2) & _M32
    x = x ^ (x >> 15)
    return x


def hash_u32(start: int, count: int, key: tuple[int, int], device) -> torch.Tensor:
    """Counter-based uint32 stream (as int64 values) for indices start..start+count-1."""
    i = torch.arange(start, start + count, dtype=torch.int64, device=device)
    k1, k2 = key
    return _mix32(_mix32((i + k1) & _M32) ^ k2)


def random_code_bytes(nbytes: int, key, device, byte_start: int = 0) -> torch.Tensor:
    """nbytes uniform random bytes (two uniform 4-bit codes each) of stream `key`."""
    assert nbytes % 4 == 0 and byte_start % 4 == 0
    v = hash_u32(byte_start // 4, nbytes // 4, key, device)
    v = torch.where(v >= 2**31, v - 2**32, v).to(torch.int32)
    return v.view(torch.uint8)  # little-endian on both host architectures


def random_scales(count: int, key, device, start: int = 0) -> torch.Tensor:
    """fp16 scales ~ U(0.002, 0.02) (rounded to fp16) of stream `key`."""
    v = hash_u32(start, count, key, device)
    u = (v >> 8).to(torch.float32) * (2.0 ** -24)          # exact, in [0, 1)
    s = torch.mul(u, torch.tensor(0.018, dtype=torch.float32, device=device))
    s = torch.add(s, torch.tensor(0.002, dtype=torch.float32, device=device))
    return s.to(torch.float16)


@dataclass
class W4Proj:
    """One 4-bit projection in the checkpoint layout (see module docstring)."""
    codes: torch.Tensor   # uint8 [rows][cols/2]
    scale: torch.Tensor   # fp16 [rows][cols/64]
    bias: torch.Tensor    # fp16 [rows][cols/64]

    @property
    def rows(self) -> int:
        return self.codes.shape[-2]

    @property
    def cols(self) -> int:
        return self.codes.shape[-1] * 2

    def to(self, device) -> "W4Proj":
        return W4Proj(self.codes.to(device), self.scale.to(device), self.bias.to(device))


@dataclass
class Expert:
    up: W4Proj            # rows = neurons, cols = hidden
    down: W4Proj          # rows = hidden, cols = neurons (checkpoint layout)
    offset: torch.Tensor  # fp32 [neurons]

    @property
    def neurons(self) -> int:
        return self.up.rows

    def to(self, device) -> "Expert":
        return Expert(self.up.to(device), self.down.to(device), self.offset.to(device))


def gen_proj(rows: int, cols: int, key_parts: tuple, device="cpu", index: int = 0) -> W4Proj:
    """Projection number `index` of stream `key_parts` (index selects an expert
    inside a stack that shares one stream, so a single expert regenerates alone)."""
    assert cols % 64 == 0 and (cols // 2) % 4 == 0
    nb = rows * cols // 2
    ng = rows * cols // 64
    codes = random_code_bytes(nb, stream_key(*key_parts, "codes"), device, index * nb)
    scale = random_scales(ng, stream_key(*key_parts, "scale"), device, index * ng)
    bias = -(scale * 8)  # exact in fp16
    return W4Proj(codes.reshape(rows, cols // 2), scale.reshape(rows, cols // 64),
                  bias.reshape(rows, cols // 64))


def code_group_sq_sums(codes: torch.Tensor) -> torch.Tensor:
    """Exact int32 sums over each group of 64 codes of (q - 8)^2, [rows][cols/64]."""
    c = codes.to(torch.int16)
    lo = (c & 15) - 8
    hi = (c >> 4) - 8
    sq = (lo * lo + hi * hi).to(torch.int32)              # [rows][cols/2]
    return sq.reshape(codes.shape[0], -1, 32).sum(dim=-1, dtype=torch.int32)


def calibrated_offsets(up: W4Proj, p, dead: np.ndarray | None = None) -> torch.Tensor:
    """fp32 offsets off_n = Phi^-1(p_n) * ||w_n||, -inf for dead neurons (CPU tensor).

    Relies on bias = -8*scale (true for every projection this module makes)."""
    sq = code_group_sq_sums(up.codes).cpu().numpy().astype(np.float64)
    sc = up.scale.cpu().numpy().astype(np.float64)
    norm2 = np.zeros(sq.shape[0], dtype=np.float64)
    for g in range(sq.shape[1]):  # fixed order: identical per row whatever the batch
        norm2 += (sc[:, g] * sc[:, g]) * sq[:, g]
    p = np.broadcast_to(np.asarray(p, dtype=np.float64), norm2.shape)
    off = ndtri(p) * np.sqrt(norm2)
    off = off.astype(np.float32)
    if dead is not None:
        off[dead] = -np.inf
    return torch.from_numpy(off)


def dead_mask(neurons: int, frac: float, *key_parts) -> np.ndarray:
    """Boolean mask of round(frac*neurons) permanently dead neurons, scattered."""
    if frac <= 0:
        return np.zeros(neurons, dtype=bool)
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(_seed_ints("dead", *key_parts))))
    m = np.zeros(neurons, dtype=bool)
    m[rng.permutation(neurons)[: int(round(frac * neurons))]] = True
    return m


def gen_expert(key_parts: tuple, neurons: int, hidden: int = HIDDEN, p: float = 0.1,
               dead_frac: float = 0.0, device="cpu", index: int = 0,
               dead_parts: tuple | None = None) -> Expert:
    """One expert (up, down, offsets) of stream `key_parts`, number `index` in its stack."""
    up = gen_proj(neurons, hidden, (*key_parts, "up"), device, index)
    down = gen_proj(hidden, neurons, (*key_parts, "down"), device, index)
    dead = dead_mask(neurons, dead_frac, *(dead_parts or key_parts), index) if dead_frac > 0 else None
    off = calibrated_offsets(up, p, dead).to(device)
    return Expert(up, down, off)


def gen_routed_stack(key_parts: tuple, n_experts: int, neurons: int, hidden: int = HIDDEN,
                     device="cpu"):
    """All routed experts' projections of one layer as stacked tensors.

    Returns (up, down) W4Proj whose tensors carry a leading expert axis; expert e
    is bit-identical to gen_proj(..., index=e) of the same stream (the stream
    position of expert e starts where expert e-1's ends)."""
    out = []
    for name, rows, cols in (("up", neurons, hidden), ("down", hidden, neurons)):
        kp = (*key_parts, name)
        nb = rows * cols // 2
        ng = rows * cols // 64
        codes = random_code_bytes(n_experts * nb, stream_key(*kp, "codes"), device, 0)
        scale = random_scales(n_experts * ng, stream_key(*kp, "scale"), device, 0)
        bias = -(scale * 8)
        out.append(W4Proj(codes.reshape(n_experts, rows, cols // 2), scale.reshape(n_experts, rows, cols // 64),
                          bias.reshape(n_experts, rows, cols // 64)))
    return out[0], out[1]


def stack_offsets(up: W4Proj, p, dead: np.ndarray | None = None) -> torch.Tensor:
    """calibrated_offsets for a stacked [E][N] up projection (CPU fp32 [E][N]);
    row for row identical to calibrated_offsets of each expert alone."""
    E, N = up.codes.shape[0], up.codes.shape[1]
    flat = W4Proj(up.codes.reshape(E * N, -1), up.scale.reshape(E * N, -1), up.bias.reshape(E * N, -1))
    d = None if dead is None else np.asarray(dead).reshape(E * N)
    return calibrated_offsets(flat, p, d).reshape(E, N)


def _rng(*parts) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(_seed_ints(*parts))))


def normal_f32(shape, *parts, mean: float = 0.0) -> torch.Tensor:
    return torch.from_numpy(_rng(*parts).normal(mean, 1.0, size=shape).astype(np.float32))


def normal_bf16(shape, *parts) -> torch.Tensor:
    return normal_f32(shape, *parts).to(torch.bfloat16)


def uniform_f64(shape, lo: float, hi: float, *parts) -> np.ndarray:
    return _rng(*parts).uniform(lo, hi, size=shape)


def shared_live_fraction(seed: int, layer: int) -> float:
    """Per-layer live fraction of the shared expert in the stacked-layer sweep, U(0.05, 0.15)."""
    return float(uniform_f64((), 0.05, 0.15, seed, "p_shared", layer))


def expert_down_h(seed: int = 0, neurons: int = N_ROUTED, p: float = 0.1) -> torch.Tensor:
    """Input of the single-expert down projection: the squared positive part of
    z ~ N(Phi^-1(p), 1), so that a fraction p of the entries is non-zero (fp32)."""
    z = _rng(seed, "expert-down", "z").normal(float(ndtri(p)), 1.0, size=neurons)
    h = np.where(z > 0.0, z * z, 0.0)
    return torch.from_numpy(h.astype(np.float32))
