"""ctypes binding of libhs (include/hs.h): argument marshalling only.

Every function here has the name of the C entry point it calls.  Tensors are
torch tensors already on the device; they are passed as raw pointers.  No
computation of the path happens in Python, and nothing falls back to the CPU:
if libhs.so is missing or fails to load, every call raises.
"""
from __future__ import annotations

import ctypes as C
import os
import re

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhs.so")
HEADER = os.path.join(os.path.dirname(PKG), "include", "hs.h")

HS_OK = 0
HS_ERR_INVALID_ARG = -1
HS_ERR_MISALIGNED = -2
HS_ERR_UNSUPPORTED_SHAPE = -3
HS_ERR_WORKSPACE = -4
HS_ERR_CUDA = -5
HS_ERR_TIMEOUT = -6
HS_FORCE_DENSE = 0x1
HS_BATCH_EXPERT_UNION = 0x2
HS_DOWN_ROW_SCALES = 0x4
HS_PREFILL_ROW_GATHER = 0x8


class HsError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status} ({hs_status_string(status)})")


class hs_w4(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("sb", C.c_void_p)]


class hs_expert(C.Structure):
    _fields_ = [("up", hs_w4), ("down_nm", hs_w4), ("up_offset", C.c_void_p), ("neurons", C.c_int)]


class hs_moe_layer(C.Structure):
    _fields_ = [("routed", C.POINTER(hs_expert)), ("n_routed", C.c_int), ("shared", C.POINTER(hs_expert)),
                ("hidden", C.c_int), ("top_k", C.c_int)]


class hs_decode_debug(C.Structure):
    _fields_ = [("topk_idx", C.c_void_p), ("topk_w", C.c_void_p), ("h", C.c_void_p), ("live_rows", C.c_void_p),
                ("live_groups", C.c_void_p), ("live_mask", C.c_void_p)]


class hs_prefill_debug(C.Structure):
    _fields_ = [("topk_idx", C.c_void_p), ("topk_w", C.c_void_p), ("tiles", C.c_void_p), ("work", C.c_void_p),
                ("live_mask", C.c_void_p), ("tile_live", C.c_void_p)]


_lib = None

_SIGS = {
    "hs_status_string": (C.c_char_p, [C.c_int]),
    "hs_device_status": (C.c_int, [C.POINTER(C.c_int)]),
    "hs_selftest_bounded_wait": (C.c_int, [C.c_longlong, C.c_void_p]),
    "hs_repack_down_nm": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                                    C.c_void_p]),
    "hs_pack_sb": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "hs_expert_down_sparse_workspace_size": (C.c_size_t, [C.c_int, C.c_int]),
    "hs_expert_down_sparse": (C.c_int, [C.c_void_p, C.POINTER(hs_w4), C.c_int, C.c_int, C.c_void_p, C.c_void_p,
                                        C.c_void_p, C.c_void_p, C.c_uint, C.c_void_p, C.c_size_t, C.c_void_p]),
    "hs_expert_down_sparse_noalloc": (C.c_int, [C.c_void_p, C.POINTER(hs_w4), C.c_int, C.c_int, C.c_void_p,
                                                C.c_void_p, C.c_void_p, C.c_void_p, C.c_uint, C.c_void_p]),
    "hs_moe_layer_decode_workspace_size": (C.c_size_t, [C.POINTER(hs_moe_layer), C.c_int]),
    "hs_moe_layer_decode": (C.c_int, [C.POINTER(hs_moe_layer), C.c_void_p, C.c_void_p, C.c_int, C.c_void_p,
                                      C.c_void_p, C.c_uint, C.POINTER(hs_decode_debug), C.c_void_p, C.c_size_t,
                                      C.c_void_p]),
    "hs_requant_down_rowscale": (C.c_int, [C.c_void_p, C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_void_p,
                                           C.c_void_p, C.c_void_p]),
    "hs_router_logits": (C.c_int, [C.c_void_p, C.c_void_p, C.c_int, C.c_int, C.c_int, C.c_void_p, C.c_void_p]),
    "hs_moe_prefill_workspace_size": (C.c_size_t, [C.POINTER(hs_moe_layer), C.c_int]),
    "hs_moe_prefill": (C.c_int, [C.POINTER(hs_moe_layer), C.c_void_p, C.c_void_p, C.c_int, C.c_void_p, C.c_void_p,
                                 C.c_uint, C.POINTER(hs_prefill_debug), C.c_void_p, C.c_size_t, C.c_void_p]),
}


def lib() -> C.CDLL:
    """The loaded libhs.so.  Raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libhs.so is not built ({LIB_PATH}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            if hasattr(L, name):
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
        _lib = L
    return _lib


def declared_functions() -> list[str]:
    """Names of the functions include/hs.h declares for export (its static
    inline helpers are compiled into the caller and are not exported)."""
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    txt = re.sub(r"^\s*static\s+inline\b.*$", "", txt, flags=re.M)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(hs_\w+)\s*\(", txt, flags=re.M)))


def hs_row_sb_words(out_dim: int) -> int:
    """Words per neuron row of a row-scale (scale, bias) array (the header's
    inline helper of the same name): one per 64 outputs, padded to 16 bytes."""
    return ((out_dim // 64) + 3) & ~3


def _p(t) -> int | None:
    """Raw device pointer of a tensor (None for None)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _check(fn: str, st: int):
    if st != HS_OK:
        raise HsError(fn, st)


def hs_status_string(status: int) -> str:
    return lib().hs_status_string(status).decode()


def hs_device_status() -> int:
    v = C.c_int(0)
    _check("hs_device_status", lib().hs_device_status(C.byref(v)))
    return v.value


def hs_selftest_bounded_wait(limit_cycles, stream=None):
    _check("hs_selftest_bounded_wait", lib().hs_selftest_bounded_wait(int(limit_cycles), _stream(stream)))


def hs_repack_down_nm(codes_om, scale_om, bias_om, out_dim, neurons, codes_nm, sb_nm, stream=None):
    _check("hs_repack_down_nm", lib().hs_repack_down_nm(_p(codes_om), _p(scale_om), _p(bias_om), out_dim, neurons,
                                                        _p(codes_nm), _p(sb_nm), _stream(stream)))


def hs_pack_sb(scale, bias, rows, groups, sb, stream=None):
    _check("hs_pack_sb", lib().hs_pack_sb(_p(scale), _p(bias), rows, groups, _p(sb), _stream(stream)))


def hs_expert_down_sparse_workspace_size(neurons, out_dim) -> int:
    return lib().hs_expert_down_sparse_workspace_size(neurons, out_dim)


def hs_expert_down_sparse(h, down_codes, down_sb, neurons, out_dim, y_bf16, y_f32=None, live_count=None, flags=0,
                          workspace=None, workspace_bytes=None, stream=None, live_idx=None):
    """One expert's sparse down projection.  The workspace must be zero-filled
    before its first use (the call leaves it so)."""
    w = hs_w4(_p(down_codes), _p(down_sb))
    nb = workspace_bytes if workspace_bytes is not None else (workspace.numel() * workspace.element_size()
                                                              if workspace is not None else 0)
    _check("hs_expert_down_sparse", lib().hs_expert_down_sparse(
        _p(h), C.byref(w), neurons, out_dim, _p(y_bf16), _p(y_f32), _p(live_idx), _p(live_count), flags,
        _p(workspace), nb, _stream(stream)))


def hs_expert_down_sparse_noalloc(h, down_codes, down_sb, neurons, out_dim, y_bf16, y_f32=None, live_count=None,
                                  flags=0, stream=None, live_idx=None):
    """hs_expert_down_sparse with the library's built-in scratch (no workspace)."""
    w = hs_w4(_p(down_codes), _p(down_sb))
    _check("hs_expert_down_sparse_noalloc", lib().hs_expert_down_sparse_noalloc(
        _p(h), C.byref(w), neurons, out_dim, _p(y_bf16), _p(y_f32), _p(live_idx), _p(live_count), flags,
        _stream(stream)))


def make_expert(up_codes, up_sb, down_codes, down_sb, offset, neurons) -> hs_expert:
    return hs_expert(hs_w4(_p(up_codes), _p(up_sb)), hs_w4(_p(down_codes), _p(down_sb)), _p(offset), neurons)


class Layer:
    """Host descriptor of one MoE layer (hs_moe_layer) built from device tensors.

    routed: list of hs_expert; shared: hs_expert or None.  Keeps the ctypes
    arrays alive for as long as the descriptor is used."""

    def __init__(self, routed: list, shared, hidden: int, top_k: int):
        self._routed = (hs_expert * len(routed))(*routed)
        self._shared = shared
        self.c = hs_moe_layer(self._routed, len(routed),
                              C.pointer(shared) if shared is not None else None, hidden, top_k)

    @property
    def ref(self):
        return C.byref(self.c)


def hs_moe_layer_decode_workspace_size(layer: Layer, batch: int) -> int:
    return lib().hs_moe_layer_decode_workspace_size(layer.ref, batch)


def hs_moe_layer_decode(layer: Layer, x_bf16, logits, batch, y_bf16, y_f32=None, flags=0, debug=None,
                        workspace=None, workspace_bytes=None, stream=None):
    nb = workspace_bytes if workspace_bytes is not None else (workspace.numel() * workspace.element_size()
                                                              if workspace is not None else 0)
    dbg = None
    if debug is not None:
        dbg = C.byref(hs_decode_debug(_p(debug.get("topk_idx")), _p(debug.get("topk_w")), _p(debug.get("h")),
                                      _p(debug.get("live_rows")), _p(debug.get("live_groups")),
                                      _p(debug.get("live_mask"))))
    _check("hs_moe_layer_decode", lib().hs_moe_layer_decode(
        layer.ref, _p(x_bf16), _p(logits), batch, _p(y_bf16), _p(y_f32), flags, dbg, _p(workspace), nb,
        _stream(stream)))


def hs_requant_down_rowscale(codes_om, scale_om, bias_om, out_dim, neurons, codes_nm, sb_row, stream=None):
    _check("hs_requant_down_rowscale", lib().hs_requant_down_rowscale(
        _p(codes_om), _p(scale_om), _p(bias_om), out_dim, neurons, _p(codes_nm), _p(sb_row), _stream(stream)))


def hs_router_logits(x_bf16, w_router, batch, hidden, n_experts, logits, stream=None):
    _check("hs_router_logits", lib().hs_router_logits(_p(x_bf16), _p(w_router), batch, hidden, n_experts,
                                                      _p(logits), _stream(stream)))


def hs_moe_prefill_workspace_size(layer: Layer, tokens: int) -> int:
    return lib().hs_moe_prefill_workspace_size(layer.ref, tokens)


def hs_moe_prefill(layer: Layer, x_bf16, logits, tokens, y_bf16, y_f32=None, flags=0, debug=None, workspace=None,
                   workspace_bytes=None, stream=None):
    nb = workspace_bytes if workspace_bytes is not None else (workspace.numel() * workspace.element_size()
                                                              if workspace is not None else 0)
    dbg = None
    if debug is not None:
        dbg = C.byref(hs_prefill_debug(_p(debug.get("topk_idx")), _p(debug.get("topk_w")), _p(debug.get("tiles")),
                                       _p(debug.get("work")), _p(debug.get("live_mask")),
                                       _p(debug.get("tile_live"))))
    _check("hs_moe_prefill", lib().hs_moe_prefill(
        layer.ref, _p(x_bf16), _p(logits), tokens, _p(y_bf16), _p(y_f32), flags, dbg, _p(workspace), nb,
        _stream(stream)))
