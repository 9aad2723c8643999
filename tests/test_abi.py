"""The C ABI (CPU): libhs.so builds, loads, exports every declared symbol, and
rejects bad arguments with the documented status codes before any GPU work."""
import ctypes as C

import pytest

from activation_sparse_moe_gb300 import build as hsbuild
from activation_sparse_moe_gb300 import hs


@pytest.fixture(scope="module")
def lib():
    hsbuild.build()
    return hs.lib()


def test_exports_every_declared_symbol(lib):
    names = hs.declared_functions()
    assert len(names) >= 8
    for n in ("hs_repack_down_nm", "hs_expert_down_sparse", "hs_moe_layer_decode", "hs_status_string"):
        assert n in names
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        s = hs.hs_status_string(code)
        assert s and s != "unknown status"
    assert hs.hs_status_string(-99) == "unknown status"


def test_down_sparse_argument_errors(lib):
    f = lib.hs_expert_down_sparse
    w = hs.hs_w4(0x10000, 0x20000)
    W = C.byref(w)
    A = 0x100000  # fake, 16-byte aligned; validation fails before it is touched
    assert f(None, W, 1856, 2688, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_INVALID_ARG
    assert f(A, W, 1856, 2688, None, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_INVALID_ARG
    assert f(A, W, 1800, 2688, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, W, 1856, 2690, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, W, 1856, 3136, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, W, 65600, 2688, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A, W, -64, 2688, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_INVALID_ARG
    assert f(A + 4, W, 1856, 2688, A, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_MISALIGNED
    assert f(A, W, 1856, 2688, A + 2, None, None, None, 0, A, 1 << 30, None) == hs.HS_ERR_MISALIGNED
    assert f(A, W, 1856, 2688, A, None, A + 2, None, 0, A, 1 << 30, None) == hs.HS_ERR_MISALIGNED
    assert f(A, W, 1856, 2688, A, None, None, A + 1, 0, A, 1 << 30, None) == hs.HS_ERR_MISALIGNED
    # flags other than HS_FORCE_DENSE belong to the layer entry points
    for fl in (hs.HS_BATCH_EXPERT_UNION, hs.HS_DOWN_ROW_SCALES):
        assert f(A, W, 1856, 2688, A, None, None, None, fl, A, 1 << 30, None) == hs.HS_ERR_INVALID_ARG
    need = hs.hs_expert_down_sparse_workspace_size(1856, 2688)
    assert need >= 2688 * 4 + 29 * 8  # one chunk's partial band per output, the group masks
    assert f(A, W, 1856, 2688, A, None, None, None, 0, A, need - 1, None) == hs.HS_ERR_WORKSPACE
    assert f(A, W, 1856, 2688, A, None, None, None, 0, None, need, None) == hs.HS_ERR_WORKSPACE
    assert hs.hs_expert_down_sparse_workspace_size(100, 2688) == 0
    assert hs.hs_expert_down_sparse_workspace_size(1856, 3136) == 0


def _layer(n_routed=4, top_k=2, hidden=256, neurons=128, shared=True, base=0x1000000):
    ex = [hs.make_expert(base, base, base, base, None, neurons) for _ in range(n_routed)]
    sh = hs.make_expert(base, base, base, base, None, 256) if shared else None
    return hs.Layer(ex, sh, hidden, top_k)


def test_layer_decode_argument_errors(lib):
    f = lib.hs_moe_layer_decode
    A = 0x200000
    L = _layer()
    need = hs.hs_moe_layer_decode_workspace_size(L, 1)
    assert need == ((4 + 2 * 2) * 256 * 4 + 255) // 256 * 256 + 256
    assert f(L.ref, A, A, 1, A, None, 0, None, A, need - 1, None) == hs.HS_ERR_WORKSPACE
    assert f(L.ref, None, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_INVALID_ARG
    assert f(L.ref, A, A, 0, A, None, 0, None, A, need, None) == hs.HS_ERR_INVALID_ARG
    assert f(L.ref, A + 8, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_MISALIGNED
    assert f(_layer(top_k=5).ref, A, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(_layer(hidden=200).ref, A, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(_layer(hidden=4096).ref, A, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(_layer(neurons=100).ref, A, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(_layer(base=0x1000008).ref, A, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_MISALIGNED
    assert f(None, A, A, 1, A, None, 0, None, A, need, None) == hs.HS_ERR_INVALID_ARG
    # mixed routed sizes are rejected
    ex = [hs.make_expert(A, A, A, A, None, 128), hs.make_expert(A, A, A, A, None, 192)]
    assert f(hs.Layer(ex, None, 256, 1).ref, A, A, 1, A, None, 0, None, A, need, None) == \
        hs.HS_ERR_UNSUPPORTED_SHAPE


def test_repack_argument_errors(lib):
    f = lib.hs_repack_down_nm
    A = 0x300000
    assert f(None, A, A, 2688, 1856, A, A, None) == hs.HS_ERR_INVALID_ARG
    assert f(A, A, A, 2688, 1800, A, A, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert f(A + 1, A, A, 2688, 1856, A, A, None) == hs.HS_ERR_MISALIGNED
    assert lib.hs_pack_sb(A, A, 0, 42, A, None) == hs.HS_ERR_INVALID_ARG
    assert lib.hs_pack_sb(A, A, 10, 42, A + 2, None) == hs.HS_ERR_MISALIGNED


def _stacked_layer(n_routed=4, top_k=2, hidden=256, neurons=128, shared=True, base=0x1000000):
    """Fake descriptors with the routed codes stacked back to back (expert e at
    base + e * neurons * hidden / 2), as the prefill requires."""
    step = neurons * hidden // 2
    ex = [hs.make_expert(base + e * step, base + e * step, base + e * step, base + e * step, None, neurons)
          for e in range(n_routed)]
    sh = hs.make_expert(base, base, base, base, None, 256) if shared else None
    return hs.Layer(ex, sh, hidden, top_k)


def test_prefill_argument_errors(lib):
    f = lib.hs_moe_prefill
    A = 0x400000
    L = _stacked_layer()
    need = hs.hs_moe_prefill_workspace_size(L, 100)
    assert need > 100 * 256 * (2 + 2 * 2)
    assert f(L.ref, A, A, 100, A, None, 0, None, A, need - 1, None) == hs.HS_ERR_WORKSPACE
    assert f(L.ref, A, A, 100, A, None, 0, None, None, need, None) == hs.HS_ERR_WORKSPACE
    assert f(L.ref, None, A, 100, A, None, 0, None, A, need, None) == hs.HS_ERR_INVALID_ARG
    assert f(L.ref, A, A, 100, None, None, 0, None, A, need, None) == hs.HS_ERR_INVALID_ARG
    assert f(L.ref, A, A, 0, A, None, 0, None, A, need, None) == hs.HS_ERR_INVALID_ARG
    assert f(L.ref, A + 2, A, 100, A, None, 0, None, A, need, None) == hs.HS_ERR_MISALIGNED
    assert f(L.ref, A, A, 4097, A, None, 0, None, A, need, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert hs.hs_moe_prefill_workspace_size(L, 4097) == 0
    # routed experts not stacked back to back, and hidden not a multiple of 128
    assert hs.hs_moe_prefill_workspace_size(_layer(), 100) == 0
    assert hs.hs_moe_prefill_workspace_size(_stacked_layer(hidden=192), 100) == 0
    # the workspace grows with the token count
    assert hs.hs_moe_prefill_workspace_size(L, 200) > need


def test_batch_decode_shape_limits(lib):
    """The CUDA-core batch kernels (2..50 tokens) take experts of at most 3712
    neurons and a hidden size that is a multiple of 128; from 51 tokens the
    prefill kernels (stacked experts) take up to 4096 neurons."""
    f = lib.hs_moe_layer_decode
    A = 0x500000
    ok = _stacked_layer(neurons=3712)
    big = _stacked_layer(neurons=4096)
    for B in (2, 9, 50):
        assert hs.hs_moe_layer_decode_workspace_size(ok, B) > 0
        assert hs.hs_moe_layer_decode_workspace_size(big, B) == 0
        assert f(big.ref, A, A, B, A, None, 0, None, A, 1 << 40, None) == hs.HS_ERR_UNSUPPORTED_SHAPE
    assert hs.hs_moe_layer_decode_workspace_size(big, 51) == hs.hs_moe_prefill_workspace_size(big, 51) > 0
    # the same limit on the shared expert
    ex = [hs.make_expert(0x1000000 + e * 128 * 128, 0x1000000, 0x1000000, 0x1000000, None, 128) for e in range(4)]
    wide_shared = hs.Layer(ex, hs.make_expert(A, A, A, A, None, 3776), 256, 2)
    assert hs.hs_moe_layer_decode_workspace_size(wide_shared, 9) == 0
    assert hs.hs_moe_layer_decode_workspace_size(_stacked_layer(hidden=192), 9) == 0
    # batch 1 takes the 4096-neuron experts
    assert hs.hs_moe_layer_decode_workspace_size(big, 1) > 0


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the built library every call raises: there is no fallback."""
    monkeypatch.setattr(hs, "LIB_PATH", str(tmp_path / "libhs.so"))
    monkeypatch.setattr(hs, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        hs.lib()
    with pytest.raises(RuntimeError, match="not built"):
        hs.hs_status_string(0)
