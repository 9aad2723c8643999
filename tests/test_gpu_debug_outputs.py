"""Every debug output of the decode and prefill calls is optional on its own.

The calls take a struct of device pointers, each of which may be NULL.  A
struct that names only the router indices, or only the router weights, must
write exactly that output and leave the results unchanged: batch-1 decode,
the small-batch decode, the batch decode on the prefill's kernels, and the
prefill itself (tile path and row gather).
"""
import pytest
import torch

import synth
from activation_sparse_moe_gb300 import hs
from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


@pytest.fixture(scope="module")
def layer():
    H, E, NR, NS, K = 256, 8, 128, 192, 3
    L = synth.layer_inputs(7, "t-dbg", 0, E, NR, NS, H, p=0.2, p_shared=0.2)
    return DeviceLayer(from_synth_stack(L.up, L.down, L.offsets), from_synth_expert(L.shared), K)


def _decode(dl, X, LG, debug):
    B, H = X.shape
    ws = torch.zeros(dl.workspace_size(B), dtype=torch.uint8, device="cuda")
    y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
    yf = torch.empty((B, H), dtype=torch.float32, device="cuda")
    hs.hs_moe_layer_decode(dl.c, X.cuda(), LG.cuda(), B, y, yf, 0, debug, ws)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    return yf.cpu()


def _prefill(dl, X, LG, debug, flags):
    T, H = X.shape
    ws = torch.zeros(dl.prefill_workspace_size(T), dtype=torch.uint8, device="cuda")
    y = torch.empty((T, H), dtype=torch.bfloat16, device="cuda")
    yf = torch.empty((T, H), dtype=torch.float32, device="cuda")
    hs.hs_moe_prefill(dl.c, X.cuda(), LG.cuda(), T, y, yf, flags, debug, ws)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    return yf.cpu()


def _check_each_alone(run, B, K):
    full = {"topk_idx": torch.full((B, K), -1, dtype=torch.int32, device="cuda"),
            "topk_w": torch.full((B, K), -1.0, dtype=torch.float32, device="cuda")}
    y_full = run(full)
    idx_only = {"topk_idx": torch.full((B, K), -1, dtype=torch.int32, device="cuda")}
    w_only = {"topk_w": torch.full((B, K), -1.0, dtype=torch.float32, device="cuda")}
    assert torch.equal(run(idx_only), y_full)
    assert torch.equal(run(w_only), y_full)
    assert torch.equal(run({}), y_full)
    assert torch.equal(idx_only["topk_idx"], full["topk_idx"])
    assert torch.equal(w_only["topk_w"], full["topk_w"])
    assert int(full["topk_idx"].min()) >= 0 and float(full["topk_w"].min()) > 0.0


@pytest.mark.parametrize("B", [1, 2, 4, 16, 64])
def test_decode_router_debug_outputs_each_alone(layer, B):
    X, LG = synth.tokens(7, "t-dbg", B, B, layer.hidden, layer.routed.E)
    _check_each_alone(lambda d: _decode(layer, X, LG, d), B, layer.top_k)


@pytest.mark.parametrize("flags", [0, hs.HS_PREFILL_ROW_GATHER], ids=["tiles", "gather"])
def test_prefill_router_debug_outputs_each_alone(layer, flags):
    T = 200
    X, LG = synth.tokens(7, "t-dbg-p", T, T, layer.hidden, layer.routed.E)
    _check_each_alone(lambda d: _prefill(layer, X, LG, d, flags), T, layer.top_k)


def _units(dl):
    return dl.shared.N // 64 + dl.top_k * (dl.routed.N // 64)


@pytest.mark.parametrize("B", [1, 2, 4, 16, 64])
def test_live_mask_request_does_not_change_results(layer, B):
    """Asking for the live masks selects, on the 9..50-token path, the kernel
    instantiation that writes them; the results are the same bits."""
    X, LG = synth.tokens(7, "t-dbg-m", B, B, layer.hidden, layer.routed.E)
    masks = torch.full((B, _units(layer)), -1, dtype=torch.int64, device="cuda")
    y_m = _decode(layer, X, LG, {"live_mask": masks})
    assert torch.equal(_decode(layer, X, LG, {}), y_m)
    assert torch.equal(_decode(layer, X, LG, None), y_m)
    assert int((masks == -1).sum()) == 0   # every word written
