"""GPU parity of the 23-layer batch-1 decode stack (the benchmark's workload).

"Skipping dead neurons..." section "Most neurons are dead in every layer": the
live fraction differs from layer to layer; the benchmark sweeps the routed
live fraction p over {0.02, 0.05, 0.1, 0.2, 0.5, 1.0} (1.0 = the dense path)
with the shared expert's fraction drawn per layer from U(0.05, 0.15).  The
layers here are built exactly as the benchmark builds them: layer l of seed
0, tag "decode-23layers", p_shared from synth.shared_live_fraction, and a sweep point's
routed offsets are the p = 0.1 offsets scaled by Phi^-1(p) / Phi^-1(0.1) (the
calibration off = Phi^-1(p) * ||w|| is linear in Phi^-1(p)).  Layers 0, 11
and 22 of the stack are checked against the oracle element by element at the
sweep's extremes, and the dense flag is bit-identical on them at p = 0.1.
"""
import dataclasses

import numpy as np
import pytest
import torch
from scipy.special import ndtri

import synth
from activation_sparse_moe_gb300.layer import DeviceLayer
from test_gpu_layer import check_layer, make_layer, run_layer

pytestmark = pytest.mark.gpu

LAYERS = (0, 11, 22)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build, hs
    build.build()
    hs.lib()


@pytest.fixture(scope="module", params=LAYERS)
def decode_layer(request):
    """Layer l of the benchmark's stack (weights generated on the GPU)."""
    l = request.param
    L = synth.layer_inputs(0, "decode-23layers", l, p=0.1, p_shared=synth.shared_live_fraction(0, l), device="cuda")
    dl = make_layer(L, 6)
    x, lg = synth.tokens(0, "decode-23layers", l, 1)
    yield l, L, dl, x, lg
    del dl, L
    torch.cuda.empty_cache()


def at_live_fraction(L, dl, p):
    """The benchmark's sweep point p: routed offsets scaled from the p = 0.1 ones."""
    ratio = float(ndtri(p) / ndtri(0.1))
    off = (L.offsets.double() * ratio).float()
    return (dataclasses.replace(L, offsets=off),
            DeviceLayer(dl.routed.with_offsets(off), dl.shared, dl.top_k))


@pytest.mark.parametrize("p", [0.02, 0.5])
def test_decode_layers_sweep_point_parity(decode_layer, p):
    l, L, dl, x, lg = decode_layer
    Lp, dlp = at_live_fraction(L, dl, p)
    y, yf, flips = check_layer(Lp, dlp, x, lg, 6, f"decode layer {l} p={p}")
    assert flips <= 2
    # the routed live fraction follows p (one token: the chosen experts' neurons
    # share the same x, so a layer's fraction scatters around p)
    _, _, d = run_layer(dlp, x, lg)
    h = d["h"].double().numpy()[synth.N_SHARED:]
    frac = float((h > 0).mean())
    assert abs(frac - p) < 0.1, (l, p, frac)


def test_decode_layers_dense_flag_bit_identical(decode_layer):
    """p = 1.0 of the sweep is the dense path on the p = 0.1 inputs: the same
    bits as the sparse call, every row read."""
    from activation_sparse_moe_gb300 import hs
    l, L, dl, x, lg = decode_layer
    y1, yf1, d1 = run_layer(dl, x, lg)
    yd, yfd, dd = run_layer(dl, x, lg, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd), l
    assert int(dd["live_rows"].item()) == synth.N_SHARED + 6 * synth.N_ROUTED
    assert torch.equal(d1["live_mask"], dd["live_mask"])
