"""Device-resident experts and layers in the library's layouts.

Takes checkpoint-layout tensors (codes, fp16 scale, fp16 bias per projection;
down projection one row per output), moves them to the GPU and converts them
with the library's own kernels: hs_pack_sb for the up projection's
(scale, bias) pairs and hs_repack_down_nm for the neuron-major down rows.
Builds the hs_expert / hs_moe_layer descriptors.  Marshalling only.
"""
from __future__ import annotations

import torch

from . import hs


def _u16(t: torch.Tensor) -> torch.Tensor:
    assert t.dtype == torch.float16
    return t.contiguous().view(torch.int16)


class DeviceExperts:
    """E experts of one shape stacked on the device in the library layouts.

    up_codes [E][N][H/2] u8, up_scale/up_bias [E][N][H/64] fp16,
    down_codes [E][H][N/2] u8 (checkpoint layout), down_scale/down_bias
    [E][H][N/64] fp16, offsets [E][N] fp32 or None."""

    def __init__(self, up_codes, up_scale, up_bias, down_codes, down_scale, down_bias, offsets=None,
                 device="cuda", stream=None, down_row_scales: bool = False):
        E, N, Hh = up_codes.shape
        H = Hh * 2
        self.E, self.N, self.H = E, N, H
        dev = torch.device(device)
        self.up_codes = up_codes.to(dev).contiguous()
        self.up_sb = torch.empty((E, N, H // 64), dtype=torch.int32, device=dev)
        us, ub = _u16(up_scale.to(dev)), _u16(up_bias.to(dev))
        hs.hs_pack_sb(us, ub, E * N, H // 64, self.up_sb, stream)
        self.dn_codes = torch.empty((E, N, H // 2), dtype=torch.uint8, device=dev)
        dc = down_codes.to(dev).contiguous()
        ds, db = _u16(down_scale.to(dev)), _u16(down_bias.to(dev))
        self.down_row_scales = down_row_scales
        if down_row_scales:
            # re-quantised with one (scale, bias) per neuron row and 64 outputs (HS_DOWN_ROW_SCALES)
            self.dn_sb = torch.empty((E, N, hs.hs_row_sb_words(H)), dtype=torch.int32, device=dev)
            for e in range(E):
                hs.hs_requant_down_rowscale(dc[e], ds[e], db[e], H, N, self.dn_codes[e], self.dn_sb[e], stream)
        else:
            self.dn_sb = torch.empty((E, N // 64, H), dtype=torch.int32, device=dev)
            for e in range(E):
                hs.hs_repack_down_nm(dc[e], ds[e], db[e], H, N, self.dn_codes[e], self.dn_sb[e], stream)
        self.offsets = None if offsets is None else offsets.to(dev, torch.float32).contiguous()

    def with_offsets(self, offsets) -> "DeviceExperts":
        """The same device weights with other pre-activation offsets [E][N] (fp32)."""
        other = object.__new__(DeviceExperts)
        other.__dict__.update(self.__dict__)
        other.offsets = None if offsets is None else offsets.to(self.up_codes.device, torch.float32).contiguous()
        return other

    def desc(self, e: int) -> hs.hs_expert:
        return hs.make_expert(self.up_codes[e], self.up_sb[e], self.dn_codes[e], self.dn_sb[e],
                              None if self.offsets is None else self.offsets[e], self.N)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.up_codes, self.up_sb, self.dn_codes, self.dn_sb))


def from_synth_stack(up, down, offsets, device="cuda", stream=None, down_row_scales=False) -> DeviceExperts:
    """DeviceExperts from stacked checkpoint-layout projections (objects with
    .codes/.scale/.bias tensors carrying a leading expert axis)."""
    return DeviceExperts(up.codes, up.scale, up.bias, down.codes, down.scale, down.bias, offsets, device, stream,
                         down_row_scales)


def from_synth_expert(ex, device="cuda", stream=None, down_row_scales=False) -> DeviceExperts:
    """A one-expert DeviceExperts from a single checkpoint-layout expert."""
    u, d = ex.up, ex.down
    return DeviceExperts(u.codes[None], u.scale[None], u.bias[None], d.codes[None], d.scale[None], d.bias[None],
                         None if ex.offset is None else ex.offset[None], device, stream, down_row_scales)


class DeviceLayer:
    """One MoE layer: routed DeviceExperts + optional shared, and its hs_moe_layer."""

    def __init__(self, routed: DeviceExperts, shared: DeviceExperts | None, top_k: int = 6):
        self.routed, self.shared, self.top_k = routed, shared, top_k
        self.hidden = routed.H
        self.c = hs.Layer([routed.desc(e) for e in range(routed.E)],
                          shared.desc(0) if shared is not None else None, routed.H, top_k)

    def workspace_size(self, batch: int = 1) -> int:
        return hs.hs_moe_layer_decode_workspace_size(self.c, batch)

    def prefill_workspace_size(self, tokens: int) -> int:
        return hs.hs_moe_prefill_workspace_size(self.c, tokens)

    def nbytes(self) -> int:
        return self.routed.nbytes() + (self.shared.nbytes() if self.shared is not None else 0)
