"""fp64 CPU oracle of the activation-sparse ReLU^2 MoE layer (test infrastructure).

Source: "Skipping dead neurons: a faster Nemotron 3.5 Lightning on Apple
silicon" (sevren.ai, "Heimr Sparse Down").  Section names below are that
page's.  Where the page is silent the plainest reading is taken and named.

What is computed, per token x (hidden size H):
  * router: the 6 largest of 128 logits are chosen ("Inside a MoE layer"); ties
    go to the lower expert index (reading); the weights are a softmax over the
    6 chosen logits only (reading: the page names no normalisation);
  * every chosen routed expert and the always-on shared expert
    ("Inside a MoE layer") widen x to their neurons with a 4-bit up projection,
    add a per-neuron offset (the synthetic workloads' calibration term), and
    apply ReLU^2, h = max(z, 0)^2 ("Transposing to skip the zeros",
    "Two projections and a switch");
  * the down projection narrows h back to H outputs, y = W_down h, summed over
    ALL neurons: the sparse method reaches the same result because the skipped
    rows are multiplied by zero ("Our way reads only the rows that fired":
    same up projection, same ReLU^2, same answer);
  * the layer output is y_shared + sum_j w_j * y_{e_j} (reading: the shared
    expert has weight 1, no routed scaling factor).
The 4-bit weights use the mlx-style affine format with one fp16 scale and
bias per group of 64 along the input axis ("The whole decode step": a scale
for every group of 64 neurons), dequantised as w = scale * q + bias in fp64
(exact for fp16 scale/bias and 4-bit q).  Packing order (reading): code of
input column 2j in the low nibble of byte j.

No blocking, fusion or reordering is done beyond what these definitions say;
matrix-vector and matrix-matrix products use numpy's fp64 matmul.
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "as_f64", "unpack_codes", "dequant", "up_preact", "relu2", "live_set",
    "down_dense", "down_dense_sequential", "down_sparse_sequential",
    "router_logits", "router_topk", "expert_forward", "moe_layer", "moe_tokens", "bf16_rne",
    "group_live", "down_required_bytes",
]


def as_f64(t) -> np.ndarray:
    """Exact widening of a torch tensor (any float dtype) or array to fp64."""
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().cpu().double().numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.float64)


def _u8(t) -> np.ndarray:
    try:
        import torch
        if isinstance(t, torch.Tensor):
            return t.detach().cpu().numpy().astype(np.uint8)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(t, dtype=np.uint8)


def unpack_codes(codes) -> np.ndarray:
    """Packed 4-bit codes [rows][cols/2] -> integer codes [rows][cols].

    Column 2j is the low nibble of byte j, column 2j+1 its high nibble."""
    b = _u8(codes)
    q = np.empty(b.shape[:-1] + (b.shape[-1] * 2,), dtype=np.int64)
    q[..., 0::2] = b & 0x0F
    q[..., 1::2] = b >> 4
    return q


def dequant(proj) -> np.ndarray:
    """Dequantised fp64 matrix [rows][cols] of a checkpoint-layout projection.

    w[r, c] = scale[r, c // 64] * q[r, c] + bias[r, c // 64].  A matrix that
    is already dense (a numpy array, e.g. a re-quantised down projection
    dequantised elsewhere) is taken as it is."""
    if isinstance(proj, np.ndarray):
        return proj.astype(np.float64)
    q = unpack_codes(proj.codes).astype(np.float64)
    s = np.repeat(as_f64(proj.scale), 64, axis=-1)
    b = np.repeat(as_f64(proj.bias), 64, axis=-1)
    return s * q + b


def up_preact(x, up, offset=None) -> np.ndarray:
    """z = W_up x + offset: the up projection of one token (x: [H]) or of many ([T][H])."""
    w = dequant(up)
    z = as_f64(x) @ w.T
    if offset is not None:
        z = z + as_f64(offset)
    return z


def relu2(z) -> np.ndarray:
    """ReLU^2: negatives (and zeros) become 0, positives are squared."""
    z = np.asarray(z, dtype=np.float64)
    return np.where(z > 0.0, z * z, 0.0)


def live_set(h) -> np.ndarray:
    """Indices of the neurons that fired, ascending: {n : h_n > 0}."""
    return np.flatnonzero(np.asarray(h) > 0.0)


def group_live(h, group: int = 64) -> np.ndarray:
    """Per group of `group` neurons: does any neuron of the group fire."""
    h = np.asarray(h)
    return (h.reshape(h.shape[:-1] + (-1, group)) > 0.0).any(axis=-1)


def down_dense(h, down) -> np.ndarray:
    """y = W_down h over all neurons (W_down: [H][neurons], checkpoint layout)."""
    return as_f64(h) @ dequant(down).T


def down_dense_sequential(h, down) -> np.ndarray:
    """The same product accumulated neuron by neuron in ascending order."""
    w = dequant(down)
    h = as_f64(h)
    y = np.zeros(w.shape[0], dtype=np.float64)
    for n in range(w.shape[1]):
        y = y + w[:, n] * h[n]
    return y


def down_sparse_sequential(h, down) -> np.ndarray:
    """The sparse form: only the live rows, in ascending order.  Equal to
    down_dense_sequential bit for bit, since every skipped term is +-0."""
    w = dequant(down)
    h = as_f64(h)
    y = np.zeros(w.shape[0], dtype=np.float64)
    for n in live_set(h):
        y = y + w[:, n] * h[n]
    return y


def router_logits(x, w_router) -> np.ndarray:
    """The router projection ("Inside a MoE layer": a router picks 6 of 128
    experts; the projection is not printed, reading: a linear map from the
    token to one logit per expert), logits[..., e] = sum_k W[e][k] x[..., k].

    x: [H] or [T][H]; w_router: [E][H].  fp64 (inputs widened exactly)."""
    return as_f64(x) @ as_f64(w_router).T


def router_topk(logits, k: int = 6):
    """Top-k experts (ties -> lower index) and softmax weights over the chosen k.

    logits: [E] or [T][E].  Returns (idx int64 [..., k] in descending logit
    order, w fp64 [..., k])."""
    l = as_f64(logits)
    idx = np.argsort(-l, axis=-1, kind="stable")[..., :k]
    sel = np.take_along_axis(l, idx, axis=-1)
    m = sel.max(axis=-1, keepdims=True)
    e = np.exp(sel - m)
    return idx, e / e.sum(axis=-1, keepdims=True)


def expert_forward(x, expert) -> dict:
    """One expert on one token: z, h, live set and y (fp64)."""
    z = up_preact(x, expert.up, expert.offset)
    h = relu2(z)
    return {"z": z, "h": h, "live": live_set(h), "y": down_dense(h, expert.down)}


def moe_layer(x, logits, routed, shared, k: int = 6) -> dict:
    """One MoE layer on one token.

    routed: callable e -> Expert (checkpoint layout); shared: Expert or None.
    Returns dict(out fp64 [H], idx, w, experts={e: expert_forward dict},
    shared=expert_forward dict or None)."""
    idx, w = router_topk(logits, k)
    out = np.zeros(as_f64(x).shape[-1], dtype=np.float64)
    sh = None
    if shared is not None:
        sh = expert_forward(x, shared)
        out = out + sh["y"]
    per = {}
    for j in range(k):
        e = int(idx[j])
        r = expert_forward(x, routed(e))
        per[e] = r
        out = out + w[j] * r["y"]
    return {"out": out, "idx": idx, "w": w, "experts": per, "shared": sh}


def moe_tokens(X, logits, routed, shared, k: int = 6) -> dict:
    """The MoE layer applied to each of T tokens (batch decode, prefill).

    X: [T][H]; logits: [T][E].  The per-token definition of moe_layer, with
    every expert's products evaluated for all of its tokens at once.
    Returns dict(out fp64 [T][H], idx [T][k], w [T][k],
    h={e: (token ids, h [t][N])}, h_shared [T][N] or None, and the
    pre-activations z={e: z [t][N]}, z_shared [T][N] or None)."""
    X = as_f64(X)
    T = X.shape[0]
    idx, w = router_topk(logits, k)
    out = np.zeros_like(X)
    hs = zs = None
    if shared is not None:
        zs = up_preact(X, shared.up, shared.offset)
        hs = relu2(zs)
        out += hs @ dequant(shared.down).T
    hmap, zmap = {}, {}
    for e in np.unique(idx):
        e = int(e)
        toks, slot = np.nonzero(idx == e)
        ex = routed(e)
        z = up_preact(X[toks], ex.up, ex.offset)
        h = relu2(z)
        y = h @ dequant(ex.down).T
        out[toks] += w[toks, slot][:, None] * y
        hmap[e] = (toks, h)
        zmap[e] = z
    return {"out": out, "idx": idx, "w": w, "h": hmap, "h_shared": hs, "z": zmap, "z_shared": zs}


_BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def bf16_rne(v) -> np.ndarray:
    """Round fp64 values to the nearest bfloat16 (ties to even), returned as fp64.

    bfloat16: 8 significant bits, exponent range of fp32 (subnormals down to 2^-133)."""
    v = np.asarray(v, dtype=np.float64)
    out = v.copy()
    fin = np.isfinite(v) & (v != 0.0)
    _, e = np.frexp(np.where(fin, v, 1.0))      # v = m * 2^e, 0.5 <= |m| < 1
    ulp = np.ldexp(1.0, np.maximum(e - 1, -126) - 7)
    r = np.round(np.where(fin, v, 0.0) / ulp) * ulp
    r = np.where(np.abs(r) > _BF16_MAX, np.copysign(np.inf, v), r)
    out[fin] = r[fin]
    return out


def down_required_bytes(h, hidden: int, group: int = 64) -> int:
    """Bytes a neuron-major sparse down projection must read for one token:
    one packed row (hidden/2 bytes) per live neuron and one (scale, bias) fp16
    pair per output for every group with a live neuron ("The whole decode
    step": a scale must be read even if one neuron of its group is alive; a
    group of 64 dead neurons costs no scales)."""
    return int(live_set(h).size * (hidden // 2) + group_live(h, group).sum() * hidden * 4)
