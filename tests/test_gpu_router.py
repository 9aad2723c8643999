"""GPU parity of hs_router_logits against the oracle, alone and chained into
the layer decode.

"Skipping dead neurons..." section "Inside a MoE layer": a router picks 6 of
128 experts for each token; the projection that produces its logits is read
as a linear map of the token's hidden state (bf16 weights and activations,
fp32 accumulation).  Calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import check_bf16_within_one_ulp, check_close
from activation_sparse_moe_gb300 import hs
from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


def run_router(X, W):
    B, H = X.shape
    E = W.shape[0]
    lg = torch.full((B, E), float("nan"), dtype=torch.float32, device="cuda")
    hs.hs_router_logits(X.cuda().contiguous(), W.cuda().contiguous(), B, H, E, lg)
    torch.cuda.synchronize()
    return lg.cpu().double().numpy()


def fp32_bound(X, W):
    """|fp32 sum - exact| <= (H + 32) u sum_k |w_k x_k| for one chain of at
    most H products and a 5-level tree of 32 partial sums (u = 2^-24)."""
    a = np.abs(oracle.as_f64(X)) @ np.abs(oracle.as_f64(W)).T
    return (X.shape[1] + 32) * 2.0 ** -24 * a


def check_logits(X, W, what):
    got = run_router(X, W)
    ref = oracle.router_logits(X, W)
    bound = fp32_bound(X, W)
    assert np.isfinite(got).all(), what
    assert (np.abs(got - ref) <= bound).all(), f"{what}: logits beyond the fp32 accumulation bound"
    # top-6 on the kernel's logits: the oracle's order, except within the bound of a tie
    for b in range(X.shape[0]):
        i_got, _ = oracle.router_topk(got[b], 6)
        i_ref, _ = oracle.router_topk(ref[b], 6)
        if not np.array_equal(i_got, i_ref):
            srt = np.sort(ref[b])[::-1]
            assert np.min(np.abs(np.diff(srt[:8]))) <= 2 * bound[b].max(), f"{what}: top-6 differs without a near tie"
    return got


@pytest.mark.parametrize("B", [1, 3, 8, 9, 64])
def test_router_logits_full_size(B):
    X, _ = synth.tokens(0, "router", B, B)
    W = synth.router_weights(0, "router", 0)
    got = check_logits(X, W, f"B={B}")
    # about N(0, 1) as the given logits of the other workloads
    assert 0.5 < got.std() < 1.5


@pytest.mark.parametrize("B,H,E", [(1, 64, 6), (2, 3072, 128), (5, 128, 13), (17, 2688, 1)])
def test_router_logits_shapes(B, H, E):
    X, _ = synth.tokens(1, "router-shape", H, B, H, E)
    W = synth.router_weights(1, "router-shape", H, E, H)
    check_logits(X, W, f"B={B} H={H} E={E}")


def test_router_logits_deterministic_and_argument_checks():
    X, _ = synth.tokens(2, "router-det", 0, 4)
    W = synth.router_weights(2, "router-det", 0)
    assert np.array_equal(run_router(X, W), run_router(X, W))
    lg = torch.empty((4, 128), dtype=torch.float32, device="cuda")
    Xc, Wc = X.cuda(), W.cuda()
    with pytest.raises(hs.HsError) as e:
        hs.hs_router_logits(Xc, Wc, 4, 2688 + 32, 128, lg)
    assert e.value.status == hs.HS_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(hs.HsError) as e:
        hs.hs_router_logits(Xc, Wc, 0, 2688, 128, lg)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    with pytest.raises(hs.HsError) as e:
        hs.hs_router_logits(Xc.view(-1)[1:], Wc, 1, 64, 1, lg)  # x 2 bytes off alignment: refused before launch
    assert e.value.status == hs.HS_ERR_MISALIGNED


@pytest.mark.parametrize("B", [1, 2])
def test_router_then_layer_decode(B):
    """Router and layer on one stream: the layer decode waits for the logits
    (programmatic dependent launch) and routes on them.  The oracle layer
    takes the kernel's fp32 logits, so the top-6 decision is made in the same
    precision on both sides; the logits themselves are checked above."""
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(4, "router-layer", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    dl = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets), from_synth_expert(L.shared), K)
    X, _ = synth.tokens(4, "router-layer", B, B, H, E)
    W = synth.router_weights(4, "router-layer", 0, E, H)
    Xc, Wc = X.cuda(), W.cuda()
    lg = torch.empty((B, E), dtype=torch.float32, device="cuda")
    y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    yf = torch.empty((B, H), dtype=torch.float32, device="cuda")
    ws = torch.zeros(dl.workspace_size(B), dtype=torch.uint8, device="cuda")
    torch.cuda.synchronize()  # inputs and workspace ready before the side stream uses them
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        lg.fill_(float("nan"))
        hs.hs_router_logits(Xc, Wc, B, H, E, lg, stream=s)
        hs.hs_moe_layer_decode(dl.c, Xc, lg, B, y, yf, 0, None, ws, stream=s)
    s.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    got_lg = lg.cpu().double().numpy()
    assert (np.abs(got_lg - oracle.router_logits(X, W)) <= fp32_bound(X, W)).all()
    ref = oracle.moe_tokens(X, got_lg, L.routed_expert, L.shared, k=K)
    yf_np = yf.cpu().double().numpy()
    check_close(yf_np, ref["out"], f"router+layer B={B}")
    for b in range(B):
        check_bf16_within_one_ulp(y.cpu()[b], ref["out"][b], f"router+layer token {b}", yf_np[b])
