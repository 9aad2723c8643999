"""The allocation-free sparse down projection (hs_expert_down_sparse_noalloc).

It serves callers that cannot give the library a workspace (a plugin whose
host framework owns every device allocation, or a path that must stay out of
the CUDA allocator).  It runs the same kernels as hs_expert_down_sparse with
scratch taken from a fixed array inside the library, so its outputs must
equal the workspace entry point's bit for bit, call after call.
Collected last on purpose: it also runs after every other GPU test.
"""
import numpy as np
import pytest
import torch

import synth
from activation_sparse_moe_gb300 import hs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


def _u16(t):
    return t.contiguous().view(torch.int16)


def _repack(down):
    H, N = down.rows, down.cols
    codes = torch.empty((N, H // 2), dtype=torch.uint8, device="cuda")
    sb = torch.empty((N // 64, H), dtype=torch.int32, device="cuda")
    hs.hs_repack_down_nm(down.codes.cuda(), _u16(down.scale.cuda()), _u16(down.bias.cuda()), H, N, codes, sb)
    return codes, sb


def _outputs(H):
    return (torch.empty(H, dtype=torch.bfloat16, device="cuda"), torch.empty(H, dtype=torch.float32, device="cuda"),
            torch.full((1,), -1, dtype=torch.int32, device="cuda"))


def _with_workspace(h, codes, sb, N, H):
    y, yf, cnt = _outputs(H)
    ws = torch.empty(hs.hs_expert_down_sparse_workspace_size(N, H), dtype=torch.uint8, device="cuda")
    hs.hs_expert_down_sparse(h, codes, sb, N, H, y, yf, cnt, 0, ws)
    torch.cuda.synchronize()
    return y.cpu(), yf.cpu().double().numpy(), int(cnt.item())


def _no_alloc(h, codes, sb, N, H):
    y, yf, cnt = _outputs(H)
    hs.hs_expert_down_sparse_noalloc(h, codes, sb, N, H, y, yf, cnt, 0)
    torch.cuda.synchronize()
    return y.cpu(), yf.cpu().double().numpy(), int(cnt.item())


def test_no_alloc_matches_workspace_entry_point_twice():
    N, H = synth.N_ROUTED, synth.HIDDEN
    h1, down = synth.single_expert_down(0)
    codes, sb = _repack(down)
    # a second input with a different live set: the shared scratch keeps the
    # first call's contents, which must not leak into the second call
    h2 = synth.config1_h(7)
    for h in (h1.cuda(), h2.cuda()):
        y_ref, yf_ref, c_ref = _with_workspace(h, codes, sb, N, H)
        y, yf, c = _no_alloc(h, codes, sb, N, H)
        assert np.array_equal(yf, yf_ref) and torch.equal(y, y_ref)
        assert c == c_ref
    assert hs.hs_device_status() == hs.HS_OK


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    A = 0x100000
    w = hs.hs_w4(A, A)
    import ctypes as C
    f = hs.lib().hs_expert_down_sparse_noalloc
    assert f(A, C.byref(w), 4160, 2688, A, None, None, 0, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, C.byref(w), 1856, 3136, A, None, None, 0, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
