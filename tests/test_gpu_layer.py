"""GPU parity of hs_moe_layer_decode (batch 1) against the oracle.

"Skipping dead neurons..." sections "Inside a MoE layer" (top-6 of 128 plus a
shared expert), "Two projections and a switch" (up, ReLU^2, down) and "Our
way reads only the rows that fired".  Calls go through the C ABI.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from _util import check_bf16_within_one_ulp, check_close, mask_bits, z_bound_cuda_core
from activation_sparse_moe_gb300 import hs
from activation_sparse_moe_gb300.layer import DeviceLayer, from_synth_expert, from_synth_stack

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


def make_layer(L: synth.LayerInputs, top_k):
    routed = from_synth_stack(L.up, L.down, L.offsets)
    shared = from_synth_expert(L.shared) if L.shared is not None else None
    return DeviceLayer(routed, shared, top_k)


def run_layer(dl: DeviceLayer, x, lg, flags=0):
    H = dl.hidden
    NS = dl.shared.N if dl.shared is not None else 0
    ws = torch.zeros(dl.workspace_size(1), dtype=torch.uint8, device="cuda")
    y = torch.empty(H, dtype=torch.bfloat16, device="cuda")
    yf = torch.empty(H, dtype=torch.float32, device="cuda")
    dbg = {"topk_idx": torch.full((dl.top_k,), -1, dtype=torch.int32, device="cuda"),
           "topk_w": torch.zeros(dl.top_k, dtype=torch.float32, device="cuda"),
           "h": torch.full((NS + dl.top_k * dl.routed.N,), -1.0, dtype=torch.float32, device="cuda"),
           "live_rows": torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           "live_groups": torch.full((1,), -1, dtype=torch.int32, device="cuda"),
           "live_mask": torch.full(((NS + dl.top_k * dl.routed.N) // 64,), -1, dtype=torch.int64, device="cuda")}
    hs.hs_moe_layer_decode(dl.c, x.reshape(-1).cuda(), lg.reshape(-1).cuda(), 1, y, yf, flags, dbg, ws)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    return y.cpu(), yf.cpu().double().numpy(), {k: v.cpu() for k, v in dbg.items()}


def check_layer(L: synth.LayerInputs, dl, x, lg, top_k, what):
    y, yf, dbg = run_layer(dl, x, lg)
    ref = oracle.moe_layer(x.reshape(-1), lg.reshape(-1), L.routed_expert, L.shared, k=top_k)
    # router: indices exact, weights to fp32 precision
    assert dbg["topk_idx"].tolist() == ref["idx"].tolist(), what
    np.testing.assert_allclose(dbg["topk_w"].double().numpy(), ref["w"], rtol=2e-6, atol=1e-7)
    # live sets: the kernel's own h > 0 equals the oracle's, except where the
    # oracle's |z| is within the CUDA-core up product's rounding bound of 0
    hk = dbg["h"].double().numpy()
    # the live-set output is exactly the kernel's own h > 0, neuron by neuron
    assert np.array_equal(mask_bits(dbg["live_mask"].numpy().view(np.uint64)), hk > 0), what
    NS = L.shared.neurons if L.shared is not None else 0
    slots = ([(L.shared, ref["shared"], 0)] if L.shared is not None else []) + [
        (L.routed_expert(int(e)), ref["experts"][int(e)], NS + j * L.up.codes.shape[1])
        for j, e in enumerate(ref["idx"])]
    flips = 0
    live_total = 0
    live_groups = 0
    for ex, r, base in slots:
        n = ex.neurons
        hg = hk[base:base + n]
        assert (hg >= 0).all()
        live_total += int((hg > 0).sum())
        live_groups += int((hg.reshape(-1, 64) > 0).any(axis=1).sum())
        mism = (hg > 0) != (r["h"] > 0)
        if mism.any():
            bound = z_bound_cuda_core(x.reshape(-1), ex.up, ex.offset)
            zmag = np.abs(r["z"])
            assert (zmag[mism] <= bound[mism]).all(), f"{what}: live-set mismatch beyond the rounding bound"
            flips += int(mism.sum())
        check_close(hg, r["h"], f"{what} h")
    assert int(dbg["live_rows"].item()) == live_total
    assert int(dbg["live_groups"].item()) == live_groups
    check_close(yf, ref["out"], f"{what} y_f32")
    check_bf16_within_one_ulp(y, ref["out"], f"{what} y_bf16", yf)
    return y, yf, flips


def test_small_layer():
    H, E, NR, NS, K = 512, 8, 128, 256, 3
    L = synth.layer_inputs(0, "t-small", 0, E, NR, NS, H, p=0.2, p_shared=0.3)
    x, lg = synth.tokens(0, "t-small", 0, 1, H, E)
    dl = make_layer(L, K)
    check_layer(L, dl, x, lg, K, "small")


def test_no_shared_top1_and_extreme_hidden():
    for H, E, NR, K in ((64, 4, 64, 1), (3072, 6, 192, 2)):
        L = synth.layer_inputs(1, "t-edge", H, E, NR, 0, H, p=0.3)
        x, lg = synth.tokens(1, "t-edge", H, 1, H, E)
        dl = make_layer(L, K)
        check_layer(L, dl, x, lg, K, f"edge H={H}")


@pytest.fixture(scope="module")
def full_layer():
    """One full-size MoE layer at live fraction 0.1 (weights generated on the GPU)."""
    L = synth.layer_inputs(0, "layer-p0.1", 0, device="cuda")
    dl = make_layer(L, 6)
    x, lg = synth.tokens(0, "layer-p0.1", 0, 1)
    return L, dl, x, lg


def test_full_layer_parity(full_layer):
    L, dl, x, lg = full_layer
    y, yf, flips = check_layer(L, dl, x, lg, 6, "full layer")
    assert flips <= 2


def test_full_layer_dense_flag_and_determinism(full_layer):
    L, dl, x, lg = full_layer
    y1, yf1, d1 = run_layer(dl, x, lg)
    y2, yf2, d2 = run_layer(dl, x, lg)
    yd, yfd, dd = run_layer(dl, x, lg, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    assert int(dd["live_rows"].item()) == 3712 + 6 * 1856
    assert torch.equal(dd["live_mask"], d1["live_mask"])  # the live set, not the rows the dense flag reads
    frac = int(d1["live_rows"].item()) / (3712 + 6 * 1856)
    assert 0.07 < frac < 0.13


def test_generator_device_independent(full_layer):
    """The GPU-generated stack equals the CPU generator for a sampled expert."""
    L, dl, x, lg = full_layer
    e = 77
    cpu = synth.gen_expert((0, "layer-p0.1", 0, "routed"), synth.N_ROUTED, index=e)
    assert torch.equal(cpu.up.codes, L.up.codes[e].cpu()) and torch.equal(cpu.down.scale, L.down.scale[e].cpu())
    assert torch.equal(cpu.offset, L.offsets[e])


def test_bounded_wait_gives_up_and_reports():
    """Failure detection without a fault: a wait that nothing completes gives
    up after its limit, the error word reads HS_ERR_TIMEOUT once, and the
    context still runs a layer decode correctly afterwards."""
    import time
    t0 = time.time()
    hs.hs_selftest_bounded_wait(20_000_000)   # ~10 ms of clock cycles
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_ERR_TIMEOUT
    assert hs.hs_device_status() == hs.HS_OK   # read and cleared
    assert time.time() - t0 < 30
    with pytest.raises(hs.HsError) as e:
        hs.hs_selftest_bounded_wait(0)
    assert e.value.status == hs.HS_ERR_INVALID_ARG
    # the context is still usable
    H, E, NR, NS, K = 256, 4, 128, 128, 2
    L = synth.layer_inputs(9, "t-after-timeout", 0, E, NR, NS, H, p=0.3, p_shared=0.3)
    X, LG = synth.tokens(9, "t-after-timeout", 0, 1, H, E)
    check_layer(L, make_layer(L, K), X[0], LG[0], K, "after timeout")


def test_up_gemv_mixed_magnitude_x_within_fixed_point_bound():
    """The up GEMV takes x as a 16-bit fixed-point copy with one exponent per
    64-input group, so inputs far below their group's maximum lose bits.
    Every group here holds one large input (64) and small ones (~2^-6), and
    every neuron is made live (offset 10 times the spread of z), so the
    kernel's z = sqrt(h) can be compared with the oracle's neuron by neuron:
    the difference stays within the bound that adds the fixed-point rounding
    (2^(E-16) per input, max |x_g| < 2^E) to the fp32 rounding."""
    from _util import z_bound_cuda_core
    H, E, NR, NS, K = 512, 4, 128, 128, 2
    L = synth.layer_inputs(11, "t-mixed", 0, E, NR, NS, H, p=0.5, p_shared=0.5)
    rng = np.random.default_rng(11)
    xs = rng.normal(0.0, 2.0 ** -6, H)
    xs[rng.integers(0, 64, H // 64) + 64 * np.arange(H // 64)] = 64.0 * rng.choice([-1.0, 1.0], H // 64)
    x = torch.from_numpy(xs.astype(np.float32)).to(torch.bfloat16)
    lg = synth.normal_f32((1, E), 11, "t-mixed", "logits")
    xv = oracle.as_f64(x)

    def live_offsets(up):
        w = oracle.dequant(up)
        return torch.from_numpy((10.0 * np.sqrt((w * w) @ (xv * xv))).astype(np.float32))

    for e in range(E):
        L.offsets[e] = live_offsets(L.routed_expert(e).up)
    L.shared = synth.Expert(L.shared.up, L.shared.down, live_offsets(L.shared.up))
    dl = make_layer(L, K)
    y, yf, dbg = run_layer(dl, x, lg)
    ref = oracle.moe_layer(x, lg.reshape(-1), L.routed_expert, L.shared, k=K)
    hk = dbg["h"].double().numpy()
    assert (hk > 0).all()
    slots = [(L.shared, ref["shared"], 0)] + [(L.routed_expert(int(e)), ref["experts"][int(e)], NS + j * NR)
                                              for j, e in enumerate(ref["idx"])]
    worst = 0.0
    for ex, r, base in slots:
        zk = np.sqrt(hk[base:base + ex.neurons])
        bound = z_bound_cuda_core(x, ex.up, ex.offset) + 2.0 ** -22 * np.abs(r["z"])
        err = np.abs(zk - r["z"])
        assert (err <= bound).all(), f"z error {err.max():.3e} beyond the fixed-point + fp32 bound"
        worst = max(worst, float((err / bound).max()))
    check_close(yf, ref["out"], "mixed-magnitude x y_f32")
    print(f"mixed-magnitude x: largest z error {worst:.3f} of its bound")
