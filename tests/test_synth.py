"""The seeded input generator (CPU): layout, reproducibility, calibration."""
import numpy as np
import torch

import oracle
import synth


def test_bias_is_minus_eight_scale_and_scale_range():
    p = synth.gen_proj(64, 2688, (0, "t", 0, "up"))
    assert torch.equal(p.bias, -(p.scale * 8))
    s = p.scale.float()
    assert float(s.min()) >= 0.002 - 1e-6 and float(s.max()) <= 0.02 + 1e-5
    assert p.codes.dtype == torch.uint8 and p.codes.shape == (64, 1344)


def test_single_expert_regenerates_its_stack_slice():
    up, down = synth.gen_routed_stack((0, "t", 3, "routed"), 3, 128, hidden=256)
    for e in range(3):
        ex = synth.gen_expert((0, "t", 3, "routed"), 128, hidden=256, index=e)
        assert torch.equal(ex.up.codes, up.codes[e]) and torch.equal(ex.down.codes, down.codes[e])
        assert torch.equal(ex.up.scale, up.scale[e]) and torch.equal(ex.down.bias, down.bias[e])
    a = synth.gen_proj(8, 256, (1, "x"))
    b = synth.gen_proj(8, 256, (1, "x"))
    c = synth.gen_proj(8, 256, (2, "x"))
    assert torch.equal(a.codes, b.codes) and not torch.equal(a.codes, c.codes)


def test_codes_look_uniform():
    p = synth.gen_proj(512, 2688, (0, "u"))
    q = oracle.unpack_codes(p.codes)
    counts = np.bincount(q.ravel(), minlength=16) / q.size
    assert np.abs(counts - 1 / 16).max() < 2e-3


def test_offsets_calibrate_live_fraction():
    """P(w_n . x + off_n > 0) = p for x ~ N(0, I): check the empirical live fraction."""
    ex = synth.gen_expert((0, "cal", 0), 1856, p=0.1)
    X = synth.normal_bf16((24, synth.HIDDEN), 0, "cal-x")
    h = oracle.relu2(oracle.up_preact(X, ex.up, ex.offset))
    frac = (h > 0).mean()
    assert abs(frac - 0.1) < 0.01, frac
    ex5 = synth.gen_expert((0, "cal", 1), 1856, p=0.5)
    h5 = oracle.relu2(oracle.up_preact(X, ex5.up, ex5.offset))
    assert abs((h5 > 0).mean() - 0.5) < 0.02


def test_dead_neurons():
    ex = synth.gen_expert((0, "dead", 0), 1856, p=0.1, dead_frac=0.3)
    dead = torch.isneginf(ex.offset)
    assert int(dead.sum()) == round(0.3 * 1856) == 557
    m = synth.dead_mask(3712, 0.3, "s")
    assert m.sum() == 1114


def test_expert_down_h():
    h = synth.expert_down_h(0)
    assert h.dtype == torch.float32 and h.shape == (1856,)
    frac = float((h > 0).float().mean())
    assert 0.08 < frac < 0.12
    assert torch.equal(h, synth.expert_down_h(0))
