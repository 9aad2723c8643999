"""GPU parity of the row-scale down layout (HS_DOWN_ROW_SCALES) against the
oracle.

"Skipping dead neurons..." section "The whole decode step": the checkpoint's
scales sit per group of 64 neurons along the output axis, so one live neuron
costs its group's scales; re-quantising with the scales along the neuron axis
removes that toll.  hs_requant_down_rowscale must produce exactly the oracle's
codes, scales and biases (the same fp32 decisions), and the batch-1 layer
decode over such weights must match the oracle's layer on the re-quantised
weights.  Calls go through the C ABI.
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


def _u16(t):
    return t.contiguous().view(torch.int16)


@pytest.mark.parametrize("H,N", [(64, 64), (128, 192), (2688, 1856), (3072, 320)])
def test_requant_kernel_equals_oracle(H, N):
    down = synth.gen_proj(H, N, (5, "requant", H, N))
    codes = torch.empty((N, H // 2), dtype=torch.uint8, device="cuda")
    sb = torch.full((N, hs.hs_row_sb_words(H)), -1, dtype=torch.int32, device="cuda")
    hs.hs_requant_down_rowscale(down.codes.cuda(), _u16(down.scale.cuda()), _u16(down.bias.cuda()), H, N, codes, sb)
    torch.cuda.synchronize()
    ref_codes, ref_s, ref_b = oracle.requant_down_rowscale(down)
    assert np.array_equal(codes.cpu().numpy(), ref_codes)
    w = sb.cpu().numpy().view(np.uint32)
    G = H // 64
    assert np.array_equal((w[:, :G] & 0xFFFF).astype(np.uint16), ref_s.view(np.uint16))
    assert np.array_equal((w[:, :G] >> 16).astype(np.uint16), ref_b.view(np.uint16))
    assert (w[:, G:] == 0).all()  # the row padding


def rowscale_expert(ex):
    """The oracle's expert with its down projection re-quantised along the
    neuron axis (a dense fp64 matrix)."""
    W = oracle.dequant_rowscale(*oracle.requant_down_rowscale(ex.down))
    return synth.Expert(ex.up, W, ex.offset)


def run_rowscale(dl, x, lg, flags=0):
    H = dl.hidden
    ws = torch.zeros(dl.workspace_size(1), dtype=torch.uint8, device="cuda")
    y = torch.empty(H, dtype=torch.bfloat16, device="cuda")
    yf = torch.empty(H, dtype=torch.float32, device="cuda")
    dbg = {"topk_idx": torch.full((dl.top_k,), -1, dtype=torch.int32, device="cuda"),
           "topk_w": torch.zeros(dl.top_k, dtype=torch.float32, device="cuda"),
           "live_rows": torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           "live_groups": torch.full((1,), -1, dtype=torch.int32, device="cuda")}
    hs.hs_moe_layer_decode(dl.c, x.reshape(-1).cuda(), lg.reshape(-1).cuda(), 1, y, yf,
                           flags | hs.HS_DOWN_ROW_SCALES, dbg, ws)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    return y.cpu(), yf.cpu().double().numpy(), {k: v.cpu() for k, v in dbg.items()}


def check_rowscale_layer(L, K, x, lg, what):
    dl = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets, down_row_scales=True),
                     from_synth_expert(L.shared, down_row_scales=True) if L.shared is not None else None, K)
    y, yf, dbg = run_rowscale(dl, x, lg)
    ref = oracle.moe_layer(x.reshape(-1), lg.reshape(-1), lambda e: rowscale_expert(L.routed_expert(e)),
                           rowscale_expert(L.shared) if L.shared is not None else None, k=K)
    assert dbg["topk_idx"].tolist() == ref["idx"].tolist(), what
    check_close(yf, ref["out"], f"{what} y_f32")
    check_bf16_within_one_ulp(y, ref["out"], f"{what} y_bf16", yf)
    return dl, y, yf, dbg


def test_rowscale_small_layer_and_no_shared():
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(6, "rowscale", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    x, lg = synth.tokens(6, "rowscale", 0, 1, H, E)
    check_rowscale_layer(L, K, x, lg, "small")
    L = synth.layer_inputs(6, "rowscale-ns", 0, 6, 192, 0, 3072, p=0.3)
    x, lg = synth.tokens(6, "rowscale-ns", 0, 1, 3072, 6)
    check_rowscale_layer(L, 2, x, lg, "H=3072, no shared")


def test_rowscale_full_layer_dense_flag_and_determinism():
    """Full-size layer at live fraction 0.1: parity, repeat and dense flag
    give the same bits, and the live counts equal those of the slab layout
    (the up projection is unchanged)."""
    L = synth.layer_inputs(0, "layer-p0.1", 0, device="cuda")
    x, lg = synth.tokens(0, "layer-p0.1", 0, 1)
    dl, y1, yf1, d1 = check_rowscale_layer(L, 6, x, lg, "full")
    y2, yf2, _ = run_rowscale(dl, x, lg)
    yd, yfd, dd = run_rowscale(dl, x, lg, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    assert int(dd["live_rows"].item()) == synth.N_SHARED + 6 * synth.N_ROUTED
    slab = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets), from_synth_expert(L.shared), 6)
    ws = torch.zeros(slab.workspace_size(1), dtype=torch.uint8, device="cuda")
    yb = torch.empty(synth.HIDDEN, dtype=torch.bfloat16, device="cuda")
    cnt = {"live_rows": torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           "live_groups": torch.full((1,), -1, dtype=torch.int32, device="cuda")}
    hs.hs_moe_layer_decode(slab.c, x.reshape(-1).cuda(), lg.reshape(-1).cuda(), 1, yb, None, 0, cnt, ws)
    torch.cuda.synchronize()
    assert int(cnt["live_rows"].item()) == int(d1["live_rows"].item())


def test_rowscale_flag_refused_by_other_entry_points():
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(7, "rowscale-refuse", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    dl = DeviceLayer(from_synth_stack(L.up, L.down, L.offsets, down_row_scales=True),
                     from_synth_expert(L.shared, down_row_scales=True), K)
    X, LG = synth.tokens(7, "rowscale-refuse", 0, 2, H, E)
    ws = torch.zeros(dl.workspace_size(2), dtype=torch.uint8, device="cuda")
    y = torch.empty((2, H), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_moe_layer_decode(dl.c, X.cuda(), LG.cuda(), 2, y, None, hs.HS_DOWN_ROW_SCALES, None, ws)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    h = torch.zeros(NR, dtype=torch.float32, device="cuda")
    wsd = torch.empty(hs.hs_expert_down_sparse_workspace_size(NR, H), dtype=torch.uint8, device="cuda")
    with pytest.raises(hs.HsError) as e:
        hs.hs_expert_down_sparse(h, dl.routed.dn_codes[0], dl.routed.dn_sb[0], NR, H, y[0], None, None,
                                 hs.HS_DOWN_ROW_SCALES, wsd)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
