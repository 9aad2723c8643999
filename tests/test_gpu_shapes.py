"""A sweep of layer shapes through every decode and prefill path, against the
oracle.

The shapes cover the ABI's corners: top-k up to its maximum of 8, n_routed
down to top-k, hidden sizes that are and are not multiples of 48 (the down
phase's two output layouts per thread), single-group experts and 4096-neuron
experts (the prefill's 64 tiles), no shared expert, and batch sizes on both
sides of each path boundary (1: batch-1 kernel; 2..8: small-batch kernel;
9..50: persistent kernel; 51 and more: the prefill's kernels).
"""
import pytest
import torch

import synth
from activation_sparse_moe_gb300 import hs
from test_gpu_batch import check_batch
from test_gpu_layer import check_layer, make_layer
from test_gpu_prefill import check_prefill

pytestmark = pytest.mark.gpu

# (hidden, routed experts, routed neurons, shared neurons, top-k)
SHAPES = [
    (128, 8, 64, 0, 8),        # top-k at its maximum, single-group experts, no shared expert
    (384, 9, 192, 64, 8),      # hidden a multiple of 48 (12 outputs per thread), n_routed just above top-k
    (640, 16, 128, 320, 4),    # hidden not a multiple of 48 (16 outputs per thread)
    (1024, 32, 256, 512, 6),
    (256, 4, 4096, 0, 2),      # 4096-neuron experts (64 tiles of 64 neurons)
]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


@pytest.fixture(scope="module", params=range(len(SHAPES)), ids=[f"H{s[0]}_E{s[1]}_N{s[2]}_S{s[3]}_K{s[4]}"
                                                                  for s in SHAPES])
def shape_layer(request):
    H, E, NR, NS, K = SHAPES[request.param]
    L = synth.layer_inputs(20 + request.param, "t-shapes", 0, E, NR, NS, H, p=0.15, p_shared=0.2, dead_frac=0.2)
    return request.param, (H, E, NR, NS, K), L, make_layer(L, K)


def test_batch1_decode(shape_layer):
    i, (H, E, NR, NS, K), L, dl = shape_layer
    x, lg = synth.tokens(20 + i, "t-shapes-b1", 0, 1, H, E)
    check_layer(L, dl, x, lg, K, f"shape {i} batch 1")


@pytest.mark.parametrize("B", [3, 9, 51])
def test_batch_decode(shape_layer, B):
    i, (H, E, NR, NS, K), L, dl = shape_layer
    if B >= 51 and H % 128:
        pytest.skip("the prefill kernels need hidden to be a multiple of 128")
    if B < 51 and max(NR, NS) > 3712:
        # the CUDA-core batch kernels take experts of at most 3712 neurons: refused, not run
        assert dl.workspace_size(B) == 0
        X, LG = synth.tokens(20 + i, "t-shapes-batch", B, B, H, E)
        y = torch.empty((B, H), dtype=torch.bfloat16, device="cuda")
        ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
        with pytest.raises(hs.HsError) as err:
            hs.hs_moe_layer_decode(dl.c, X.cuda(), LG.cuda(), B, y, None, workspace=ws)
        assert err.value.status == hs.HS_ERR_UNSUPPORTED_SHAPE
        return
    X, LG = synth.tokens(20 + i, "t-shapes-batch", B, B, H, E)
    check_batch(L, dl, X, LG, K, f"shape {i} B={B}", flips_allowed=8)


@pytest.mark.parametrize("T", [1, 130])
def test_prefill(shape_layer, T):
    i, (H, E, NR, NS, K), L, dl = shape_layer
    if H % 128:
        pytest.skip("the prefill kernels need hidden to be a multiple of 128")
    X, LG = synth.tokens(20 + i, "t-shapes-prefill", T, T, H, E)
    check_prefill(L, dl, X, LG, K, f"shape {i} T={T}")
