"""GPU parity of hs_moe_prefill against the oracle.

"Skipping dead neurons..." sections "A whole prompt at once", "Sorted by
expert", "Per token sparse, per prompt dense" and "What we do instead": the
prompt's tokens are routed one by one, grouped by expert, and each expert's
up projection, ReLU^2 and down projection run as matrix products; the result
is the per-token MoE layer (oracle.moe_tokens).  The full-size prompt: 2048
tokens, top-6 of 128 plus the shared expert, 30% of every expert's neurons
permanently dead, p = 0.1 on the rest.

The tile skip must not change the result: the sparse call equals the
HS_FORCE_DENSE call bit for bit.  Live sets are checked element by element:
each (token, slot, neuron) of the kernel's live mask equals the oracle's
h > 0 except neurons whose oracle |z| lies within the rounding bound of the
fp16-operand products; every token tile's multiplied 64-neuron tiles equal
the union of its tokens' masks, and the skip and work counts follow from
those masks exactly.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import check_bf16_rounding, check_close, check_token_live_masks, mask_bits, plan_ksteps
from activation_sparse_moe_gb300 import hs
from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack

pytestmark = pytest.mark.gpu

TILE = 128   # tokens per token tile of the library's prefill


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


def make_layer(L, top_k):
    routed = from_synth_stack(L.up, L.down, L.offsets)
    shared = from_synth_expert(L.shared) if L.shared is not None else None
    return DeviceLayer(routed, shared, top_k)


def units_of(dl):
    NS = dl.shared.N if dl.shared is not None else 0
    return NS // 64 + dl.top_k * (dl.routed.N // 64)


def max_tiles(dl, T):
    return dl.routed.E + (T * dl.top_k + TILE - 1) // TILE + (T + TILE - 1) // TILE


def run_prefill(dl, X, LG, flags=0, masks=True):
    T, H = X.shape
    ws = torch.zeros(dl.prefill_workspace_size(T), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    yf = torch.empty((T, H), dtype=torch.float32, device="cuda")
    dbg = {"topk_idx": torch.full((T, dl.top_k), -1, dtype=torch.int32, device="cuda"),
           "topk_w": torch.zeros((T, dl.top_k), dtype=torch.float32, device="cuda"),
           "tiles": torch.full((2,), -1, dtype=torch.int32, device="cuda"),
           "work": torch.full((3,), -1, dtype=torch.int64, device="cuda")}
    if masks:
        dbg["live_mask"] = torch.full((T, units_of(dl)), -1, dtype=torch.int64, device="cuda")
        dbg["tile_live"] = torch.full((max_tiles(dl, T),), -1, dtype=torch.int64, device="cuda")
    hs.hs_moe_prefill(dl.c, X.cuda(), LG.cuda(), T, y, yf, flags, dbg, ws)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    return y.cpu(), yf.cpu().double().numpy(), {k: v.cpu() for k, v in dbg.items()}


def kernel_tiles(dl, idx, words):
    """The library's token tiles rebuilt from the routing (the routed experts
    with tokens ascending, each expert's tokens in order cut into tiles of
    TILE, then the shared expert's tokens), with, per tile, the union over its
    tokens of the kernel's own live masks: (n_tokens, group words [NK],
    union-live neurons, NK)."""
    T, K = idx.shape
    NS = dl.shared.N if dl.shared is not None else 0
    NGs, NGr = NS // 64, dl.routed.N // 64
    out = []
    for e in range(dl.routed.E):
        toks, slots = np.nonzero(idx == e)
        for r in range(0, len(toks), TILE):
            w = np.zeros(NGr, np.uint64)
            for b, j in zip(toks[r:r + TILE], slots[r:r + TILE]):
                w |= words[b, NGs + j * NGr:NGs + (j + 1) * NGr]
            out.append((len(toks[r:r + TILE]), w, NGr))
    if NS:
        for r in range(0, T, TILE):
            w = np.bitwise_or.reduce(words[r:r + TILE, :NGs], axis=0)
            out.append((min(TILE, T - r), w, NGs))
    return out


def check_tiles_from_masks(dl, dbg, what, dense=False, gather=False):
    """Each tile's multiplied 64-neuron tiles are exactly the groups where the
    union of its tokens' masks has a live neuron (all of them with the dense
    flag); the skip and work counts follow.  With the row gather the down
    product runs the k-steps of each tile's plan instead (plan_ksteps of the
    union words): 'skipped' counts the k-steps saved against one per group."""
    words = dbg["live_mask"].numpy().view(np.uint64)
    tl = dbg["tile_live"].numpy().view(np.uint64)
    tiles = kernel_tiles(dl, dbg["topk_idx"].numpy(), words)
    skipped = total = union = execd = dense_w = 0
    for i, (nt, w, NK) in enumerate(tiles):
        gl = (w != 0)
        want = sum(1 << int(j) for j in np.flatnonzero(gl)) if not dense else (1 << NK) - 1
        assert int(tl[i]) == want, (what, i, hex(int(tl[i])), hex(want))
        total += NK
        nks = plan_ksteps([int(v) for v in w]) if gather and not dense else int(bin(want).count("1"))
        skipped += NK - nks
        union += nt * int(mask_bits(w[None])[0].sum())
        execd += nt * 64 * nks
        dense_w += nt * 64 * NK
    assert [int(v) for v in dbg["tiles"]] == [skipped, total], what
    assert [int(v) for v in dbg["work"]] == [union, execd, dense_w], what
    return skipped


def check_prefill(L, dl, X, LG, K, what, flips_allowed=4, flags=0):
    y, yf, dbg = run_prefill(dl, X, LG, flags=flags)
    ref = oracle.moe_tokens(X, LG, L.routed_expert, L.shared, k=K)
    assert np.array_equal(dbg["topk_idx"].numpy(), ref["idx"]), what
    np.testing.assert_allclose(dbg["topk_w"].double().numpy(), ref["w"], rtol=2e-6, atol=1e-7)
    rel, mx = check_close(yf, ref["out"], f"{what} y_f32")
    ulps = check_bf16_rounding(y, yf, ref["out"], what)
    words = dbg["live_mask"].numpy().view(np.uint64)
    flips = check_token_live_masks(words, X, ref, L.shared, L.routed_expert, dl.routed.N, K, "fp16", what)
    print(f"{what}: rel-L2 {rel:.2e} max-abs/max {mx:.2e} bf16 max ulps from RNE(oracle) {ulps:.0f}, "
          f"live-set flips within the fp16 bound {flips}")
    n_neurons = X.shape[0] * ((L.shared.neurons if L.shared is not None else 0) + K * dl.routed.N)
    assert flips <= flips_allowed + n_neurons // 2000, (what, flips)
    check_tiles_from_masks(dl, dbg, what, gather=bool(flags & hs.HS_PREFILL_ROW_GATHER))
    return y, yf, dbg


def cluster_dead(L, n_groups, seed=0):
    """Kill whole 64-neuron groups of every routed expert (offset -inf) so that
    the tile skip has work to do (the oracle reads the same offsets)."""
    rng = np.random.default_rng(seed)
    E, N = L.offsets.shape
    for e in range(E):
        for g in rng.choice(N // 64, size=n_groups, replace=False):
            L.offsets[e, 64 * g:64 * (g + 1)] = -np.inf


GATHER = [0, hs.HS_PREFILL_ROW_GATHER]


@pytest.mark.parametrize("flags", GATHER, ids=["tiles", "gather"])
@pytest.mark.parametrize("T", [1, 37, 300])
def test_small_prefill(T, flags):
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(0, "t-prefill", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    X, LG = synth.tokens(0, "t-prefill", T, T, H, E)
    check_prefill(L, make_layer(L, K), X, LG, K, f"small T={T} flags={flags}", flags=flags)


@pytest.mark.parametrize("flags", GATHER, ids=["tiles", "gather"])
def test_multi_tile_experts_and_clustered_dead(flags):
    """More than 256 tokens per expert (several token tiles), the shared expert
    over 4 tiles, and whole dead 64-neuron groups that the skip must find."""
    H, E, NR, NS, K = 256, 4, 256, 192, 2
    L = synth.layer_inputs(2, "t-prefill-mt", 0, E, NR, NS, H, p=0.05, p_shared=0.2)
    cluster_dead(L, 2, seed=2)
    T = 900
    X, LG = synth.tokens(2, "t-prefill-mt", 0, T, H, E)
    y, yf, dbg = check_prefill(L, make_layer(L, K), X, LG, K, f"multi-tile flags={flags}", flags=flags)
    assert int(dbg["tiles"][0]) >= 2 * E * 2   # every routed tile skips at least the dead groups


@pytest.mark.parametrize("flags", GATHER, ids=["tiles", "gather"])
def test_no_shared_with_ties_and_ragged_neurons(flags):
    """No shared expert, tied logits, a neuron count that is not a multiple of
    128 (the last 128-neuron block is half empty)."""
    H, E, NR, K = 128, 6, 192, 2
    L = synth.layer_inputs(1, "t-prefill-ns", 0, E, NR, 0, H, p=0.3, dead_frac=0.3)
    X, LG = synth.tokens(1, "t-prefill-ns", 0, 50, H, E)
    LG[3, :] = 0.5
    check_prefill(L, make_layer(L, K), X, LG, K, f"no shared, ties flags={flags}", flags=flags)


def test_row_gather_deterministic_dense_flag_and_scattered_dead():
    """The row gather on scattered dead neurons (no 64-neuron group is dead
    for a whole tile, so the tile skip saves nothing and the gather saves the
    k-steps of the dead rows): repeat calls give the same bits; its result
    agrees with the tile path within the oracle's bar (the k-steps group the
    fp32 sums differently); with HS_FORCE_DENSE the flag is ignored and the
    call equals the plain dense call bit for bit."""
    H, E, NR, NS, K = 256, 4, 512, 256, 2
    L = synth.layer_inputs(5, "t-prefill-g", 0, E, NR, NS, H, p=0.1, p_shared=0.1, dead_frac=0.4)
    dl = make_layer(L, K)
    X, LG = synth.tokens(5, "t-prefill-g", 0, 700, H, E)
    G = hs.HS_PREFILL_ROW_GATHER
    y1, yf1, d1 = check_prefill(L, dl, X, LG, K, "gather, scattered dead", flags=G)
    y2, yf2, d2 = run_prefill(dl, X, LG, flags=G)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    yt, yft, dt = run_prefill(dl, X, LG)
    assert int(dt["tiles"][0]) == 0 and int(d1["tiles"][0]) > 0
    assert torch.equal(d1["live_mask"], dt["live_mask"])
    np.testing.assert_allclose(yf1, yft, rtol=0, atol=1e-4 * np.abs(yft).max())
    yd, yfd, dd = run_prefill(dl, X, LG, flags=hs.HS_FORCE_DENSE)
    ydg, yfdg, ddg = run_prefill(dl, X, LG, flags=hs.HS_FORCE_DENSE | G)
    assert np.array_equal(yfd, yfdg) and torch.equal(yd, ydg)
    assert [int(v) for v in ddg["tiles"]] == [int(v) for v in dd["tiles"]]


def test_dense_flag_bit_identical_and_deterministic():
    H, E, NR, NS, K = 256, 4, 256, 192, 2
    L = synth.layer_inputs(3, "t-prefill-d", 0, E, NR, NS, H, p=0.05, p_shared=0.2)
    cluster_dead(L, 1, seed=3)
    dl = make_layer(L, K)
    X, LG = synth.tokens(3, "t-prefill-d", 0, 400, H, E)
    y1, yf1, d1 = run_prefill(dl, X, LG)
    y2, yf2, d2 = run_prefill(dl, X, LG)
    yd, yfd, dd = run_prefill(dl, X, LG, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    assert int(dd["tiles"][0]) == 0 and int(d1["tiles"][0]) > 0
    assert int(dd["tiles"][1]) == int(d1["tiles"][1])
    # the live sets do not depend on the flag; the dense call multiplies every tile
    assert torch.equal(d1["live_mask"], dd["live_mask"]) and torch.equal(d1["live_mask"], d2["live_mask"])
    check_tiles_from_masks(dl, d1, "sparse")
    check_tiles_from_masks(dl, dd, "dense flag", dense=True)


def test_prefill_argument_errors():
    H, E, NR, NS, K = 256, 4, 128, 128, 2
    L = synth.layer_inputs(4, "t-prefill-err", 0, E, NR, NS, H)
    dl = make_layer(L, K)
    X, LG = synth.tokens(4, "t-prefill-err", 0, 8, H, E)
    x, lg = X.cuda(), LG.cuda()
    y = torch.empty((8, H), dtype=torch.bfloat16, device="cuda")
    ws = torch.zeros(dl.prefill_workspace_size(8), dtype=torch.uint8, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_moe_prefill(dl.c, x, lg, 8, y, workspace=ws, workspace_bytes=ws.numel() - 1)
    assert e.value.status == hs.HS_ERR_WORKSPACE
    with pytest.raises(hs.HsError) as e:
        hs.hs_moe_prefill(dl.c, x, lg, 0, y, workspace=ws)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    assert dl.prefill_workspace_size(4097) == 0
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK


@pytest.fixture(scope="module")
def prefill_2048():
    """The full-size layer, 30% permanently dead, p = 0.1 on the rest, 2048 tokens."""
    L = synth.layer_inputs(0, "prefill-2048", 0, p=0.1, p_shared=0.1, dead_frac=0.3, device="cuda")
    X, LG = synth.tokens(0, "prefill-2048", 0, 2048)
    return L, make_layer(L, 6), X, LG


@pytest.mark.parametrize("flags", GATHER, ids=["tiles", "gather"])
def test_prefill_2048_sampled_parity(prefill_2048, flags):
    """Full size, in the launch configuration the bench times; the oracle
    evaluates a sample of tokens one by one (each token's output depends on
    that token alone)."""
    L, dl, X, LG = prefill_2048
    y, yf, dbg = run_prefill(dl, X, LG, flags=flags)
    rng = np.random.default_rng(5)
    sample = np.sort(rng.choice(X.shape[0], size=16, replace=False))
    ref = oracle.moe_tokens(X[sample], LG[sample], L.routed_expert, L.shared, k=6)
    assert np.array_equal(dbg["topk_idx"].numpy()[sample], ref["idx"])
    rel, mx = check_close(yf[sample], ref["out"], "prefill 2048 sampled y_f32")
    ulps = check_bf16_rounding(y[sample], yf[sample], ref["out"], "prefill 2048 sampled")
    words = dbg["live_mask"].numpy().view(np.uint64)
    flips = check_token_live_masks(words[sample], X[sample], ref, L.shared, L.routed_expert, synth.N_ROUTED, 6,
                                   "fp16", "prefill 2048 sampled")
    print(f"prefill 2048 sampled: rel-L2 {rel:.2e} max-abs/max {mx:.2e} bf16 max ulps {ulps:.0f} flips {flips}")
    assert flips <= 4 + len(sample) * (synth.N_SHARED + 6 * synth.N_ROUTED) // 2000
    gather = bool(flags & hs.HS_PREFILL_ROW_GATHER)
    skipped = check_tiles_from_masks(dl, dbg, "prefill 2048", gather=gather)
    print(f"prefill 2048 flags={flags}: skipped k-steps {skipped}")
    if gather:   # the scattered 30% dead rows leave about a quarter of the k-steps out
        assert skipped > int(dbg["tiles"][1]) // 5
    # every (expert, token tile) pair is counted once: 58-tile shared expert + 29 tiles per routed tile
    counts = np.bincount(dbg["topk_idx"].numpy().ravel(), minlength=128)
    tiles = int(sum((c + TILE - 1) // TILE for c in counts)) * (synth.N_ROUTED // 64)
    tiles += ((2048 + TILE - 1) // TILE) * (synth.N_SHARED // 64)
    assert int(dbg["tiles"][1]) == tiles
    assert np.isfinite(yf).all()


def test_prefill_2048_dense_flag_equal(prefill_2048):
    L, dl, X, LG = prefill_2048
    y1, yf1, d1 = run_prefill(dl, X, LG, masks=False)
    yd, yfd, dd = run_prefill(dl, X, LG, flags=hs.HS_FORCE_DENSE, masks=False)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    assert int(dd["tiles"][0]) == 0


@pytest.mark.parametrize("flags", GATHER, ids=["tiles", "gather"])
def test_prefill_2048_layer_at_max_tokens(prefill_2048, flags):
    """The largest prompt chunk the library takes (4096 tokens: 24,576 routed
    pairs, 32 shared-expert tiles) on the full-size layer: sampled tokens
    (the first, the last and random ones; each routed expert's last tile is
    ragged) against the oracle, every (expert, token tile) pair counted once."""
    L, dl, _, _ = prefill_2048
    T = 4096
    assert dl.prefill_workspace_size(T) > 0 and dl.prefill_workspace_size(T + 1) == 0
    X, LG = synth.tokens(0, "prefill-max", 0, T)
    y, yf, dbg = run_prefill(dl, X, LG, flags=flags)
    rng = np.random.default_rng(6)
    sample = np.unique(np.concatenate([[0, T - 1], rng.choice(T, size=10, replace=False)]))
    ref = oracle.moe_tokens(X[sample], LG[sample], L.routed_expert, L.shared, k=6)
    assert np.array_equal(dbg["topk_idx"].numpy()[sample], ref["idx"])
    rel, mx = check_close(yf[sample], ref["out"], "4096 tokens sampled y_f32")
    check_bf16_rounding(y[sample], yf[sample], ref["out"], "4096 tokens sampled")
    words = dbg["live_mask"].numpy().view(np.uint64)
    check_token_live_masks(words[sample], X[sample], ref, L.shared, L.routed_expert, synth.N_ROUTED, 6, "fp16",
                           "4096 tokens sampled")
    check_tiles_from_masks(dl, dbg, "4096 tokens", gather=bool(flags & hs.HS_PREFILL_ROW_GATHER))
    counts = np.bincount(dbg["topk_idx"].numpy().ravel(), minlength=128)
    tiles = int(sum((c + TILE - 1) // TILE for c in counts)) * (synth.N_ROUTED // 64)
    tiles += (T // TILE) * (synth.N_SHARED // 64)
    assert int(dbg["tiles"][1]) == tiles
    assert np.isfinite(yf).all()


@pytest.mark.parametrize("flags", GATHER, ids=["tiles", "gather"])
def test_prefill_2048_repeated_calls_bit_identical(prefill_2048, flags):
    """Determinism under repetition: the full-size prefill called 16 times on
    the same inputs (fresh and reused workspaces alternating) gives the same
    bits every time."""
    L, dl, X, LG = prefill_2048
    T, H = X.shape
    Xc, LGc = X.cuda(), LG.cuda()
    ws_keep = torch.zeros(dl.prefill_workspace_size(T), dtype=torch.uint8, device="cuda")
    ref = None
    for i in range(16):
        ws = ws_keep if i % 2 else torch.zeros_like(ws_keep)
        yf = torch.empty((T, H), dtype=torch.float32, device="cuda")
        y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        hs.hs_moe_prefill(dl.c, Xc, LGc, T, y, yf, flags, None, ws)
        torch.cuda.synchronize()
        if ref is None:
            ref = yf.clone()
        else:
            bad = (yf != ref).any(dim=1).nonzero().flatten().tolist()
            assert not bad, f"call {i}: {len(bad)} tokens differ from the first call"
    assert hs.hs_device_status() == hs.HS_OK
