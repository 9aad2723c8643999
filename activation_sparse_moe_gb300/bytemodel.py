"""Bytes the activation-sparse path must move (the roofline numerator).

"Skipping dead neurons..." (sevren.ai): each projection is read once per
decode step ("Two projections and a switch"); with the down weights stored
by neuron, a dead row is never read ("Our way reads only the rows that
fired"); a group of 64 neurons with a live neuron costs its scales, a fully
dead group none ("The whole decode step").  Scales and biases are fp16.
"""
from __future__ import annotations


def w4_projection_bytes(rows: int, cols: int, group: int = 64) -> int:
    """Packed codes plus one fp16 scale and one fp16 bias per group."""
    return rows * cols // 2 + (rows * cols // group) * 4


def up_bytes(neurons: int, hidden: int, with_offsets: bool = True) -> int:
    return w4_projection_bytes(neurons, hidden) + (neurons * 4 if with_offsets else 0)


def down_sparse_bytes(live_rows: int, live_groups: int, hidden: int) -> int:
    """Neuron-major down projection: one row per live neuron, one (scale, bias)
    slab of `hidden` pairs per group with a live neuron."""
    return live_rows * (hidden // 2) + live_groups * hidden * 4


def decode_layer_bytes(hidden: int, expert_neurons: list[int], live_rows: int, live_groups: int,
                       n_routed: int, batch: int = 1) -> int:
    """Required bytes of one layer decode call: dense up projections of the
    experts that run, sparse down rows/slabs, activations in and out, logits."""
    up = sum(up_bytes(n, hidden) for n in expert_neurons)
    io = batch * (hidden * 2 + n_routed * 4 + hidden * 2)
    return up + down_sparse_bytes(live_rows, live_groups, hidden) + io


def second_copy_bytes(layers: int, n_routed: int, routed_neurons: int, shared_neurons: int, hidden: int) -> int:
    """Bytes of one extra (checkpoint-layout) copy of every down projection."""
    return layers * (n_routed * w4_projection_bytes(hidden, routed_neurons) +
                     w4_projection_bytes(hidden, shared_neurons))
