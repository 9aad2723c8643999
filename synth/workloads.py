"""The synthetic workloads, built from the seeded generator.

  single_expert_down  one routed expert's down projection and h = relu(z)^2,
                      z ~ N(Phi^-1(0.1), 1) (about 10% live), 1856 -> 2688
  layer_inputs        one MoE layer: 128 routed experts (1856 neurons) and a
                      shared expert (3712), offsets calibrated to live
                      fraction p (routed) and p_shared; optionally a fraction
                      of every expert's neurons permanently dead (offset -inf)
  tokens              x ~ N(0, 1) bf16 [batch][hidden] and logits ~ N(0, 1)
                      fp32 [batch][n_experts]

Sizes and distributions follow the page's model (section "Inside a MoE
layer": hidden 2688, 128 routed experts of 1856 neurons, top-6, a 3712-neuron
shared expert); the live fractions stand in for the page's measured ones.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

from .gen import (HIDDEN, N_EXPERTS, N_ROUTED, N_SHARED, Expert, W4Proj, expert_down_h, dead_mask, gen_expert,
                  gen_proj, gen_routed_stack, normal_bf16, normal_f32, stack_offsets)

__all__ = ["LayerInputs", "layer_inputs", "tokens", "router_weights", "single_expert_down"]


@dataclass
class LayerInputs:
    up: W4Proj            # stacked [E][N][H/2] ...
    down: W4Proj          # stacked [E][H][N/2] ... (checkpoint layout)
    offsets: torch.Tensor  # CPU fp32 [E][N]
    shared: Expert | None
    dead: np.ndarray | None  # [E][N] bool or None

    @property
    def n_experts(self) -> int:
        return self.up.codes.shape[0]

    def routed_expert(self, e: int, device="cpu") -> Expert:
        """Expert e as a standalone checkpoint-layout Expert (for the oracle)."""
        u = W4Proj(self.up.codes[e].to(device), self.up.scale[e].to(device), self.up.bias[e].to(device))
        d = W4Proj(self.down.codes[e].to(device), self.down.scale[e].to(device), self.down.bias[e].to(device))
        return Expert(u, d, self.offsets[e].to(device))


def layer_inputs(seed: int, tag: str, layer: int, n_experts: int = N_EXPERTS, routed_neurons: int = N_ROUTED,
                 shared_neurons: int = N_SHARED, hidden: int = HIDDEN, p: float = 0.1, p_shared: float = 0.1,
                 dead_frac: float = 0.0, device="cpu") -> LayerInputs:
    kp = (seed, tag, layer)
    up, down = gen_routed_stack((*kp, "routed"), n_experts, routed_neurons, hidden, device)
    dead = None
    if dead_frac > 0:
        dead = np.stack([dead_mask(routed_neurons, dead_frac, *kp, "routed", e) for e in range(n_experts)])
    off = stack_offsets(up, p, dead)
    shared = None
    if shared_neurons:
        shared = gen_expert((*kp, "shared"), shared_neurons, hidden, p_shared, dead_frac, device, 0)
        shared = Expert(shared.up, shared.down, shared.offset.cpu())
    return LayerInputs(up, down, off, shared, dead)


def tokens(seed: int, tag: str, layer: int, batch: int, hidden: int = HIDDEN, n_experts: int = N_EXPERTS):
    """x [batch][hidden] bf16 and logits [batch][n_experts] fp32 (CPU)."""
    x = normal_bf16((batch, hidden), seed, tag, layer, "x")
    lg = normal_f32((batch, n_experts), seed, tag, layer, "logits")
    return x, lg


def router_weights(seed: int, tag: str, layer: int, n_experts: int = N_EXPERTS, hidden: int = HIDDEN):
    """Router projection W [n_experts][hidden] bf16 with entries N(0, 1/hidden),
    so that the logits of x ~ N(0, 1) are about N(0, 1) like the given ones."""
    return (normal_f32((n_experts, hidden), seed, tag, layer, "router") / float(np.sqrt(hidden))).to(torch.bfloat16)


def single_expert_down(seed: int = 0, neurons: int = N_ROUTED, hidden: int = HIDDEN, p: float = 0.1,
                       device="cpu"):
    """(h fp32 [neurons], down W4Proj in checkpoint layout [hidden][neurons])."""
    down = gen_proj(hidden, neurons, (seed, "expert-down", "down"), device)
    return expert_down_h(seed, neurons, p), down
