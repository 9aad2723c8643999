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


# ------------------------------------------------------------------ live sets
def mask_bits(words) -> np.ndarray:
    """64-bit live-mask words [..., units] -> bool [..., units * 64] (bit r of
    word u = neuron 64u + r of that slot)."""
    w = np.asarray(words).astype(np.uint64)
    bits = (w[..., None] >> np.arange(64, dtype=np.uint64)) & np.uint64(1)
    return bits.reshape(w.shape[:-1] + (w.shape[-1] * 64,)).astype(bool)


def _abs_terms(up, x):
    """Per neuron: sum_k (|s| q + |b|) |x_k| and sum_k |w_nk|, and per-group
    sums of |w| (the magnitudes every rounding of the up product scales)."""
    q = oracle.unpack_codes(up.codes).astype(np.float64)
    s = np.repeat(np.abs(oracle.as_f64(up.scale)), 64, axis=-1)
    b = np.repeat(np.abs(oracle.as_f64(up.bias)), 64, axis=-1)
    xa = np.abs(oracle.as_f64(x))
    w = np.abs(oracle.dequant(up))
    return (s * q + b) @ xa, w @ xa, w


def z_bound_cuda_core(x, up, offset=None) -> np.ndarray:
    """Per neuron, an upper bound of |z_kernel - z_oracle| for the CUDA-core
    up product: x as a 16-bit fixed-point copy per 64-input group (an element
    is off by at most 2^(E-16), max|x_g| < 2^E), integer dot products (exact),
    the group's scale and bias applied and the groups summed in fp32
    ((H + 64) 2^-24 of the magnitudes involved), the offset added in fp32."""
    xf = oracle.as_f64(x)
    H = xf.shape[-1]
    split, _, w = _abs_terms(up, xf)
    mx = np.abs(xf).reshape(-1, 64).max(axis=1)
    E = np.where(mx > 0, np.floor(np.log2(np.where(mx > 0, mx, 1.0))) + 1, -100)
    fixed = w.reshape(w.shape[0], -1, 64).sum(axis=2) @ np.ldexp(1.0, (E - 16).astype(int))
    off = 0.0 if offset is None else np.abs(oracle.as_f64(offset))
    return 2.0 * ((H + 64) * 2.0 ** -24 * split + fixed + 2.0 ** -24 * off)


def z_bound_fp16_operands(x, up, offset=None) -> np.ndarray:
    """The same for the tensor-core products: the weight dequantised to fp16
    by one rounding (2^-11 relative, 2^-25 absolute below fp16's normal
    range), x converted bf16 -> fp16 (exact in the normal range, 2^-25
    below), fp32 accumulation in the tensor core ((H + 64) 2^-23 of
    sum |w||x|), the offset added in fp32."""
    xf = oracle.as_f64(x)
    H = xf.shape[-1]
    _, wx, w = _abs_terms(up, xf)
    off = 0.0 if offset is None else np.abs(oracle.as_f64(offset))
    rnd = 2.0 ** -11 * wx + 2.0 ** -25 * (w.sum(axis=1) + np.abs(xf).sum())
    return 2.0 * (rnd + (H + 64) * 2.0 ** -23 * wx + 2.0 ** -24 * off)


def live_in_precision(z, kind) -> np.ndarray:
    """The oracle's live decision taken in the kernel's precision: h = z^2
    (z > 0) rounded to fp32 ("fp32", CUDA-core kernels) or to fp16 ("fp16",
    the tensor-core kernels store h as fp16; a positive z below about
    2^-12.5 gives h = 0, a dead neuron).  h > 0 decides."""
    zz = np.where(z > 0, z * z, 0.0)
    return (zz.astype(np.float16 if kind == "fp16" else np.float32) > 0)


def check_token_live_masks(words, X, ref, shared, routed_expert, NR, K, kind, what):
    """Element-wise live-set parity of a batch call: the kernel's live mask of
    every (token, slot, neuron) equals the oracle's {h > 0}, except neurons
    whose oracle |z| lies within the kind's rounding bound ("fp32": CUDA-core
    kernels, "fp16": tensor-core kernels), which may flip.  words: [B][Ut]
    uint64 from the call's live_mask output (shared groups first, then the
    slots in topk order); shared: the shared Expert or None; routed_expert:
    descriptor index -> Expert.  The oracle's side of the decision is
    live_in_precision (h rounded as the kernel stores it).  Returns the
    number of flipped neurons."""
    bound_fn = z_bound_cuda_core if kind == "fp32" else z_bound_fp16_operands
    got = mask_bits(np.asarray(words))
    X = oracle.as_f64(X)
    B = X.shape[0]
    NS = shared.neurons if shared is not None else 0
    flips = 0
    for b in range(B):
        slots = []
        if NS:
            slots.append((shared, ref["z_shared"][b], ref["h_shared"][b], 0))
        for j in range(K):
            e = int(ref["idx"][b][j])
            toks, h = ref["h"][e]
            r = int(np.flatnonzero(toks == b)[0])
            slots.append((routed_expert(e), ref["z"][e][r], h[r], NS + j * NR))
        for ex, z, h, base in slots:
            n = ex.neurons
            mism = got[b, base:base + n] != live_in_precision(z, kind)
            if mism.any():
                bound = bound_fn(X[b], ex.up, ex.offset)
                bad = np.abs(z[mism]) > bound[mism]
                assert not bad.any(), (f"{what}: token {b}: live-set mismatch beyond the {kind} bound at "
                                       f"neurons {np.flatnonzero(mism)[bad][:8]}, |z| {np.abs(z[mism])[bad][:4]}")
                flips += int(mism.sum())
    return flips


def union_counts_from_masks(words, idx, NS, NR, K):
    """Rows and 64-neuron groups of the per-expert union of the kernel's own
    live masks (each expert once, the shared expert over every token)."""
    got = np.asarray(words).astype(np.uint64)
    B = got.shape[0]
    NGs, NGr = NS // 64, NR // 64
    per = {}
    for b in range(B):
        if NS:
            per["s"] = per.get("s", np.zeros(NGs, np.uint64)) | got[b, :NGs]
        for j in range(K):
            e = int(idx[b][j])
            per[e] = per.get(e, np.zeros(NGr, np.uint64)) | got[b, NGs + j * NGr:NGs + (j + 1) * NGr]
    rows = sum(int(mask_bits(v).sum()) for v in per.values())
    groups = sum(int((v != 0).sum()) for v in per.values())
    return rows, groups


def plan_ksteps(union_words) -> int:
    """Down-product k-steps of one token tile under the prefill's row gather,
    from the tile's union-live words (uint64 [NG], bit i of word g = neuron
    64 g + i live for some token of the tile).  The rule, restated from its
    description: each group's live neurons padded to a multiple of 8 entries;
    k-steps of 64 entries holding at most two groups (a third group closes
    the k-step, whose tail stays padding); a plan of more k-steps than
    groups gives way to one k-step per group."""
    NG = len(union_words)
    ks, fill, groups = 0, 0, 0
    for w in union_words:
        c = bin(int(w)).count("1")
        if c == 0:
            continue
        left = -(-c // 8) * 8
        if fill > 0 and groups == 2:
            ks, fill, groups = ks + 1, 0, 0
        first = True
        while left:
            if fill == 0:
                groups = 1
            elif first:
                groups = 2
            first = False
            take = min(64 - fill, left)
            fill += take
            left -= take
            if fill == 64:
                ks, fill, groups = ks + 1, 0, 0
    if fill:
        ks += 1
    return ks if ks <= NG else NG
