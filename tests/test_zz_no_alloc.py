"""The allocation-free sparse down projection (hs_expert_down_sparse_noalloc).

It serves callers that cannot give the library a workspace (a plugin whose
host framework owns every device allocation, or a path that must stay out of
the CUDA allocator).  It runs the same kernel as hs_expert_down_sparse with
scratch taken from a fixed array inside the library, so its outputs must
equal the workspace entry point's bit for bit, call after call, and meet the
oracle's bar like it.  Collected last on purpose: it also runs after every
other GPU test.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import check_bf16_within_one_ulp, check_close
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


def _outputs(N, H):
    return (torch.empty(H, dtype=torch.bfloat16, device="cuda"), torch.empty(H, dtype=torch.float32, device="cuda"),
            torch.full((1,), -1, dtype=torch.int32, device="cuda"),
            torch.full((N,), -1, dtype=torch.int32, device="cuda"))


def _result(y, yf, cnt, idx):
    c = int(cnt.item())
    return y.cpu(), yf.cpu().double().numpy(), c, idx.cpu().numpy()[:c]


def _with_workspace(h, codes, sb, N, H):
    y, yf, cnt, idx = _outputs(N, H)
    ws = torch.zeros(hs.hs_expert_down_sparse_workspace_size(N, H), dtype=torch.uint8, device="cuda")
    hs.hs_expert_down_sparse(h, codes, sb, N, H, y, yf, cnt, 0, ws, live_idx=idx)
    torch.cuda.synchronize()
    return _result(y, yf, cnt, idx)


def _no_alloc(h, codes, sb, N, H):
    y, yf, cnt, idx = _outputs(N, H)
    hs.hs_expert_down_sparse_noalloc(h, codes, sb, N, H, y, yf, cnt, 0, live_idx=idx)
    torch.cuda.synchronize()
    return _result(y, yf, cnt, idx)


@pytest.mark.parametrize("H,N", [(synth.HIDDEN, synth.N_ROUTED), (3072, 4096), (256, 65536), (64, 64)])
def test_no_alloc_matches_workspace_entry_point_twice(H, N):
    """The single-expert shape (one pass, the scratch untouched), experts
    wider than one 32-group chunk that keep their partial sums and counters
    in the scratch (4096 neurons x 3072 outputs, and 65536 neurons, the
    largest the scratch holds: 32 chunks per band), and the smallest shape:
    two inputs with different live sets in a row (the shared scratch keeps
    the first call's contents, which must not leak into the second), each
    bit-equal to the workspace entry point and within the oracle's bar, with
    the oracle's live set."""
    if (H, N) == (synth.HIDDEN, synth.N_ROUTED):
        h1, down = synth.single_expert_down(0)
        h2 = synth.expert_down_h(7)
    else:
        down = synth.gen_proj(H, N, (4, "noalloc", H, N))
        rng = np.random.default_rng(H + N)
        h1 = torch.from_numpy(oracle.relu2(rng.normal(-1.2815516, 1.0, N)).astype(np.float32))
        h2 = torch.from_numpy(oracle.relu2(rng.normal(-0.5, 1.0, N)).astype(np.float32))
    codes, sb = _repack(down)
    for h in (h1, h2):
        hd = h.cuda().float().contiguous()
        y_ref, yf_ref, c_ref, l_ref = _with_workspace(hd, codes, sb, N, H)
        y, yf, c, li = _no_alloc(hd, codes, sb, N, H)
        assert np.array_equal(yf, yf_ref) and torch.equal(y, y_ref)
        assert c == c_ref and np.array_equal(li, l_ref)
        hn = h.double().numpy()
        assert np.array_equal(li, oracle.live_set(hn))
        ref = oracle.down_dense(hn, down)
        check_close(yf, ref, f"no-alloc {H}x{N}")
        check_bf16_within_one_ulp(y, ref, f"no-alloc {H}x{N}", yf)
    assert hs.hs_device_status() == hs.HS_OK


def test_no_alloc_rejects_shapes_beyond_its_scratch():
    A = 0x100000
    w = hs.hs_w4(A, A)
    f = hs.lib().hs_expert_down_sparse_noalloc
    assert f(A, C.byref(w), 65600, 2688, A, None, None, None, 0, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, C.byref(w), 1856, 3136, A, None, None, None, 0, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, C.byref(w), 1856, 2688, A, None, None, None, hs.HS_BATCH_EXPERT_UNION, None) == hs.HS_ERR_INVALID_ARG
