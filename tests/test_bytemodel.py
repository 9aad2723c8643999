"""Byte model pinned to the page's own figures ("Skipping dead neurons...")."""
import numpy as np

import oracle
from activation_sparse_moe_gb300 import bytemodel as bm


def test_shared_projection_is_5_6_mb():
    """Section "Two projections and a switch": each projection is 5.6 MB of 4-bit weights."""
    b = bm.w4_projection_bytes(3712, 2688)
    assert b == 5_612_544
    assert round(b / 1e6, 1) == 5.6


def test_second_down_copy_is_8_4_gb():
    """Sections "The weights now face the wrong way." / "Two obvious answers, both costly":
    a second copy of the down weights costs 8.4 GB over the 23 MoE layers."""
    b = bm.second_copy_bytes(23, 128, 1856, 3712, 2688)
    assert b == 8_390_753_280
    assert round(b / 1e9, 1) == 8.4


def test_down_bytes_agree_with_oracle_count():
    rng = np.random.default_rng(0)
    h = oracle.relu2(rng.normal(-1.28, 1, 1856))
    live = len(oracle.live_set(h))
    groups = int(oracle.group_live(h).sum())
    assert bm.down_sparse_bytes(live, groups, 2688) == oracle.down_required_bytes(h, 2688)


def test_layer_bytes_at_p0_1():
    # dense up of shared + 6 routed experts, offsets included
    up = bm.up_bytes(3712, 2688) + 6 * bm.up_bytes(1856, 2688)
    assert up == 22_450_176 + 59_392
    full = bm.decode_layer_bytes(2688, [3712] + [1856] * 6, 14848, 232, 128)
    assert full == up + 14848 * 1344 + 232 * 10752 + 2688 * 4 + 512
