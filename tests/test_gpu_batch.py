"""GPU parity of hs_moe_layer_decode with batch > 1 against the oracle.

"Skipping dead neurons..." sections "Inside a MoE layer" and "Sorted by
expert": each token routes on its own; the tokens are grouped by expert and
each expert reads the union of its tokens' live rows.  The full-size layer at
batch 2..64, with 30% of every expert's neurons permanently dead, p = 0.1 on the rest.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import (check_bf16_rounding, check_bf16_within_one_ulp, check_close, check_token_live_masks,
                   union_counts_from_masks)
from activation_sparse_moe_gb300 import hs
from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack

pytestmark = pytest.mark.gpu


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
    """Live-mask words per token: shared groups, then top_k slots of routed groups."""
    NS = dl.shared.N if dl.shared is not None else 0
    return NS // 64 + dl.top_k * (dl.routed.N // 64)


def run_batch(dl, X, LG, flags=0):
    B, H = X.shape
    ws = torch.zeros(dl.workspace_size(B), dtype=torch.uint8, device="cuda")
    assert ws.numel() > 0
    y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    yf = torch.empty((B, H), dtype=torch.float32, device="cuda")
    dbg = {"topk_idx": torch.full((B, dl.top_k), -1, dtype=torch.int32, device="cuda"),
           "topk_w": torch.zeros((B, dl.top_k), dtype=torch.float32, device="cuda"),
           "live_rows": torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           "live_groups": torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           # sentinel: every word must be written (an all-ones group is impossible here)
           "live_mask": torch.full((B, units_of(dl)), -1, dtype=torch.int64, device="cuda")}
    hs.hs_moe_layer_decode(dl.c, X.cuda(), LG.cuda(), B, y, yf, flags, dbg, ws)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    return y.cpu(), yf.cpu().double().numpy(), {k: v.cpu() for k, v in dbg.items()}


PREFILL_MIN_BATCH = 51  # from here on the decode runs on the prefill's tensor-core kernels


def on_prefill_kernels(B, flags=0):
    return B >= PREFILL_MIN_BATCH and not (flags & hs.HS_BATCH_EXPERT_UNION)


def check_batch(L, dl, X, LG, K, what, flips_allowed=4, flags=0, prefill=None, routed_expert=None):
    """prefill: whether the call runs on the prefill's kernels (by default the
    library's rule for stacked layers); routed_expert: the oracle's expert of
    each descriptor index (by default the stack's).

    Live sets are checked element by element: every (token, slot, neuron) of
    the kernel's live mask equals the oracle's h > 0, except neurons whose
    oracle |z| is within the rounding bound of the path's arithmetic (fp32 on
    the CUDA-core kernels, fp16 operands on the tensor-core ones), of which
    at most flips_allowed (plus 5 per 10^4 neurons on the tensor-core path,
    whose fp16 operands move z by a few 10^-4 of sum |w x|) may flip; the
    oracle's decision is taken on h rounded as the kernel stores it (fp32 or
    fp16); the rows and groups the call read equal the union of its own masks
    exactly."""
    routed_expert = routed_expert or L.routed_expert
    y, yf, dbg = run_batch(dl, X, LG, flags=flags)
    ref = oracle.moe_tokens(X, LG, routed_expert, L.shared, k=K)
    assert np.array_equal(dbg["topk_idx"].numpy(), ref["idx"]), what
    np.testing.assert_allclose(dbg["topk_w"].double().numpy(), ref["w"], rtol=2e-6, atol=1e-7)
    check_close(yf, ref["out"], f"{what} y_f32")
    on_tc = on_prefill_kernels(X.shape[0], flags) if prefill is None else prefill
    if on_tc:
        # fp16 operands: the prefill's output contract
        check_bf16_rounding(y, yf, ref["out"], what)
    else:
        for b in range(X.shape[0]):
            check_bf16_within_one_ulp(y[b], ref["out"][b], f"{what} token {b}", yf[b])
    words = dbg["live_mask"].numpy().view(np.uint64)
    NR = dl.routed.N
    flips = check_token_live_masks(words, X, ref, L.shared, routed_expert, NR, K, "fp16" if on_tc else "fp32", what)
    n_neurons = X.shape[0] * ((L.shared.neurons if L.shared is not None else 0) + K * NR)
    assert flips <= flips_allowed + (n_neurons // 2000 if on_tc else 0), (what, flips)
    print(f"{what}: live-set flips within the rounding bound {flips} of {n_neurons} neurons")
    NS = L.shared.neurons if L.shared is not None else 0
    rows, groups = union_counts_from_masks(words, ref["idx"], NS, NR, K)
    assert int(dbg["live_rows"].item()) == rows, (what, int(dbg["live_rows"].item()), rows)
    assert int(dbg["live_groups"].item()) == groups, (what, int(dbg["live_groups"].item()), groups)
    return y, yf, dbg


@pytest.mark.parametrize("B", [2, 5, 8, 50, 51, 96, 200])
def test_small_batch(B):
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(0, "t-batch", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    X, LG = synth.tokens(0, "t-batch", B, B, H, E)
    check_batch(L, make_layer(L, K), X, LG, K, f"small B={B}")


def test_small_batch_no_shared_with_ties():
    H, E, NR, K = 256, 6, 64, 2
    L = synth.layer_inputs(1, "t-batch-ns", 0, E, NR, 0, H, p=0.3, dead_frac=0.3)
    X, LG = synth.tokens(1, "t-batch-ns", 0, 4, H, E)
    LG[1, :] = 0.5  # all tied: experts 0 and 1 by the index rule
    check_batch(L, make_layer(L, K), X, LG, K, "no shared, ties")


def single_token_decodes(dl, X, LG):
    """Each token of the batch decoded alone (batch 1)."""
    H = X.shape[1]
    ws = torch.zeros(dl.workspace_size(1), dtype=torch.uint8, device="cuda")
    out = []
    for b in range(X.shape[0]):
        y = torch.empty(H, dtype=torch.bfloat16, device="cuda")
        yf = torch.empty(H, dtype=torch.float32, device="cuda")
        hs.hs_moe_layer_decode(dl.c, X[b].cuda(), LG[b].cuda(), 1, y, yf, 0, None, ws)
        torch.cuda.synchronize()
        out.append((y.cpu(), yf.cpu().double().numpy()))
    return out


@pytest.mark.parametrize("B,H,E,NR,NS,K", [(2, 512, 8, 128, 256, 3), (3, 3072, 6, 192, 0, 2),
                                           (4, 512, 8, 128, 256, 3), (5, 512, 8, 128, 256, 3),
                                           (8, 512, 8, 128, 256, 3), (9, 512, 8, 128, 256, 3),
                                           (16, 3072, 6, 192, 0, 2)])
def test_batch_rows_equal_single_token_decode(B, H, E, NR, NS, K):
    """Batching changes no token's result: every unit adds each token's terms
    in the same order as the batch-1 kernel (rows live only for another token
    add +0), so each row of a batch decode equals that token decoded alone,
    bit for bit (B <= 8: units numbered before routing; B > 8: the ticketed
    units)."""
    L = synth.layer_inputs(2, "t-batch-eq", H, E, NR, NS, H, p=0.2, p_shared=0.3)
    X, LG = synth.tokens(2, "t-batch-eq", B, B, H, E)
    dl = make_layer(L, K)
    y, yf, _ = check_batch(L, dl, X, LG, K, f"B={B} H={H}")
    for b, (y1, yf1) in enumerate(single_token_decodes(dl, X, LG)):
        assert np.array_equal(yf[b], yf1), f"token {b}: batch row differs from its batch-1 decode"
        assert torch.equal(y[b], y1)


@pytest.mark.parametrize("B", [2, 3, 4, 5, 7, 8])
def test_small_path_every_token_on_the_same_experts(B):
    """All tokens route alike: with B <= 4 each routed unit holds all the
    tokens (3 tokens: a unit with an idle token lane, and the shared expert in
    units of 2 and 1); with 5, 7 and 8 each expert's tokens fill two units
    (token groups of 4 and the rest), whose live masks the counts must unite,
    and each row still equals its batch-1 decode."""
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(3, "t-batch-same", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    X, LG = synth.tokens(3, "t-batch-same", 0, B, H, E)
    LG[:] = LG[0].clone()
    dl = make_layer(L, K)
    y, yf, dbg = check_batch(L, dl, X, LG, K, f"same experts B={B}")
    assert len(np.unique(dbg["topk_idx"].numpy())) == K
    for b, (y1, yf1) in enumerate(single_token_decodes(dl, X, LG)):
        assert np.array_equal(yf[b], yf1) and torch.equal(y[b], y1)


@pytest.fixture(scope="module")
def batch_layer():
    """The full-size layer, 30% permanently dead, p = 0.1 on the rest."""
    L = synth.layer_inputs(0, "batch-dead0.3", 0, p=0.1, p_shared=0.1, dead_frac=0.3, device="cuda")
    return L, make_layer(L, 6)


@pytest.mark.parametrize("B", [2, 3, 4, 6, 8, 16, 32, 64])
def test_batch_layer_parity(batch_layer, B):
    L, dl = batch_layer
    X, LG = synth.tokens(0, "batch-dead0.3", B, B)
    check_batch(L, dl, X, LG, 6, f"batch layer B={B}", flips_allowed=8)


@pytest.mark.parametrize("B", [8, 64])
def test_batch_layer_parity_expert_union_path(batch_layer, B):
    """HS_BATCH_EXPERT_UNION: every expert reads the union of all its tokens'
    live rows once (banded kernels); same oracle bar, and the union count is
    the same as the default path's."""
    L, dl = batch_layer
    X, LG = synth.tokens(0, "batch-dead0.3", B, B)
    y1, yf1, d1 = check_batch(L, dl, X, LG, 6, f"batch layer B={B} expert union", flips_allowed=8,
                              flags=hs.HS_BATCH_EXPERT_UNION)
    y2, yf2, d2 = run_batch(dl, X, LG)
    r1, r2 = int(d1["live_rows"].item()), int(d2["live_rows"].item())
    g1, g2 = int(d1["live_groups"].item()), int(d2["live_groups"].item())
    if on_prefill_kernels(B):  # the default path's fp16 products: near-zero neurons may flip
        assert abs(r1 - r2) <= 8 + r1 // 100 and abs(g1 - g2) <= 8
    else:                      # the same integer up products: the same live sets
        assert r1 == r2 and g1 == g2


def test_batch_layer_dense_flag_and_determinism(batch_layer):
    L, dl = batch_layer
    X, LG = synth.tokens(0, "batch-dead0.3", 8, 8)
    y1, yf1, d1 = run_batch(dl, X, LG)
    y2, yf2, d2 = run_batch(dl, X, LG)
    yd, yfd, dd = run_batch(dl, X, LG, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    ntouched = len(np.unique(d1["topk_idx"].numpy()))
    assert int(dd["live_rows"].item()) == ntouched * synth.N_ROUTED + synth.N_SHARED
    assert int(d1["live_rows"].item()) < int(dd["live_rows"].item())
    # the same on the banded path
    f = hs.HS_BATCH_EXPERT_UNION
    yu, yfu, du = run_batch(dl, X, LG, flags=f)
    yud, yfud, dud = run_batch(dl, X, LG, flags=f | hs.HS_FORCE_DENSE)
    assert np.array_equal(yfu, yfud) and torch.equal(yu, yud)
    assert int(dud["live_rows"].item()) == ntouched * synth.N_ROUTED + synth.N_SHARED


def test_batch_layer_small_path_dense_flag_and_determinism(batch_layer):
    """B = 3 (one unit per expert, no route kernel): repeatable, dense flag
    gives the same bits, and each row equals the token decoded alone."""
    L, dl = batch_layer
    X, LG = synth.tokens(0, "batch-dead0.3", 3, 3)
    y1, yf1, d1 = run_batch(dl, X, LG)
    y2, yf2, d2 = run_batch(dl, X, LG)
    yd, yfd, dd = run_batch(dl, X, LG, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    ntouched = len(np.unique(d1["topk_idx"].numpy()))
    assert int(dd["live_rows"].item()) == ntouched * synth.N_ROUTED + synth.N_SHARED
    for b, (ys, yfs) in enumerate(single_token_decodes(dl, X, LG)):
        assert np.array_equal(yf1[b], yfs) and torch.equal(y1[b], ys)


@pytest.mark.parametrize("B,flags", [(1, 0), (2, 0), (3, 0), (8, 0), (16, 0), (8, hs.HS_BATCH_EXPERT_UNION), (56, 0)])
def test_graph_capture_equals_eager(B, flags):
    """The layer decode captured in a CUDA graph (as a serving loop replays
    it) gives the eager call's bits, replay after replay, on every path:
    batch 1, 2..8 tokens (units numbered before routing), the ticketed units
    (16 tokens), the expert-union kernels and (56 tokens) the prefill's
    tensor-core kernels."""
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(8, "t-graph", 0, E, NR, NS, H, p=0.2, p_shared=0.3, dead_frac=0.3)
    dl = make_layer(L, K)
    X, LG = synth.tokens(8, "t-graph", B, B, H, E)
    Xc, LGc = X.cuda(), LG.cuda()
    ws = torch.zeros(dl.workspace_size(B), dtype=torch.uint8, device="cuda")
    y_e = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    yf_e = torch.empty((B, H), dtype=torch.float32, device="cuda")
    y_g = torch.empty_like(y_e)
    yf_g = torch.empty_like(yf_e)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        hs.hs_moe_layer_decode(dl.c, Xc, LGc, B, y_e, yf_e, flags, None, ws, stream=s)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        hs.hs_moe_layer_decode(dl.c, Xc, LGc, B, y_g, yf_g, flags, None, ws, stream=s)
    for _ in range(3):
        y_g.zero_()
        yf_g.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(yf_g, yf_e) and torch.equal(y_g, y_e)
    assert hs.hs_device_status() == hs.HS_OK


def test_batch64_on_prefill_kernels_dense_flag_and_determinism(batch_layer):
    """B = 64 runs on the prefill's tensor-core kernels: repeatable, and the
    dense flag (no 64-neuron tile skipped) gives the same bits."""
    L, dl = batch_layer
    X, LG = synth.tokens(0, "batch-dead0.3", 64, 64)
    y1, yf1, d1 = run_batch(dl, X, LG)
    y2, yf2, _ = run_batch(dl, X, LG)
    yd, yfd, _ = run_batch(dl, X, LG, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)


def permuted_layer(L, K, pi):
    """The stacked experts handed to the library in the order pi (descriptor e
    is stack expert pi[e]): the experts no longer sit at uniform strides, so
    the kernels take each expert's pointers from the descriptor table (as for
    experts allocated one by one), and the prefill's kernels, which need one
    tensor map over a uniform stack, do not take the layer."""
    dl = make_layer(L, K)
    dl.c = hs.Layer([dl.routed.desc(int(pi[e])) for e in range(dl.routed.E)], dl.shared.desc(0), dl.hidden, K)
    return dl, (lambda e: L.routed_expert(int(pi[e])))


@pytest.mark.parametrize("B", [1, 3, 8, 16, 64])
def test_experts_not_stacked_uniformly(B):
    """Batch 1, the small-batch kernel, the ticketed kernel and, at 64 tokens
    (the CUDA-core kernels' largest batch, the prefill refusing the layer),
    the ticketed kernel again, against the oracle with the same permutation;
    the prefill entry point refuses the layer and batches above 64 are
    refused."""
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(9, "t-nonuniform", 0, E, NR, NS, H, p=0.2, p_shared=0.3, dead_frac=0.3)
    pi = np.random.default_rng(9).permutation(E)
    assert not np.array_equal(pi, np.arange(E))
    dl, routed_expert = permuted_layer(L, K, pi)
    X, LG = synth.tokens(9, "t-nonuniform", B, B, H, E)
    check_batch(L, dl, X, LG, K, f"non-uniform B={B}", prefill=False, routed_expert=routed_expert)
    if B == 64:
        assert dl.prefill_workspace_size(64) == 0
        assert dl.workspace_size(65) == 0
        y = torch.empty((65, H), dtype=torch.bfloat16, device="cuda")
        X65, LG65 = synth.tokens(9, "t-nonuniform", 65, 65, H, E)
        ws = torch.zeros(dl.workspace_size(64), dtype=torch.uint8, device="cuda")
        with pytest.raises(hs.HsError) as e:
            hs.hs_moe_layer_decode(dl.c, X65.cuda(), LG65.cuda(), 65, y, None, 0, None, ws)
        assert e.value.status == hs.HS_ERR_UNSUPPORTED_SHAPE
        with pytest.raises(hs.HsError) as e:
            hs.hs_moe_prefill(dl.c, X65.cuda(), LG65.cuda(), 65, y, workspace=ws)
        assert e.value.status == hs.HS_ERR_UNSUPPORTED_SHAPE
        torch.cuda.synchronize()
        assert hs.hs_device_status() == hs.HS_OK


@pytest.mark.parametrize("B", [8, 64])
def test_batch_layer_row_gather_flag(batch_layer, B):
    """HS_PREFILL_ROW_GATHER reaches the prefill kernels that a batch of 51 or
    more tokens runs on (same oracle bar, the same live sets, the same bits as
    the prefill entry point called with the flag); below 51 tokens it is
    ignored (the same bits as without it)."""
    L, dl = batch_layer
    X, LG = synth.tokens(0, "batch-dead0.3", B, B)
    G = hs.HS_PREFILL_ROW_GATHER
    y, yf, d = check_batch(L, dl, X, LG, 6, f"batch layer B={B} row gather flag", flips_allowed=8, flags=G)
    y0, yf0, d0 = run_batch(dl, X, LG)
    assert torch.equal(d["live_mask"], d0["live_mask"])
    if on_prefill_kernels(B):
        T, H = X.shape
        ws = torch.zeros(dl.prefill_workspace_size(T), dtype=torch.uint8, device="cuda")
        yp = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
        yfp = torch.empty((T, H), dtype=torch.float32, device="cuda")
        hs.hs_moe_prefill(dl.c, X.cuda(), LG.cuda(), T, yp, yfp, G, None, ws)
        torch.cuda.synchronize()
        assert np.array_equal(yf, yfp.cpu().double().numpy()) and torch.equal(y, yp.cpu())
    else:
        assert np.array_equal(yf, yf0) and torch.equal(y, y0)
