"""GPU parity of the repacker and of hs_expert_down_sparse against the oracle.

Single-expert activation-sparse down projection ("Skipping dead neurons...",
section "Our way reads only the rows that fired").  All calls go through the
C ABI (libhs.so) via the ctypes binding.
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from _util import check_bf16_within_one_ulp, check_close, dequant_neuron_major
from activation_sparse_moe_gb300 import hs

pytestmark = pytest.mark.gpu
GOLD = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from activation_sparse_moe_gb300 import build
    build.build()
    hs.lib()


def _u16(t):
    return t.contiguous().view(torch.int16)


def repack(down: synth.W4Proj):
    H, N = down.rows, down.cols
    codes = torch.empty((N, H // 2), dtype=torch.uint8, device="cuda")
    sb = torch.empty((N // 64, H), dtype=torch.int32, device="cuda")
    hs.hs_repack_down_nm(down.codes.cuda(), _u16(down.scale.cuda()), _u16(down.bias.cuda()), H, N, codes, sb)
    return codes, sb


def run_down(h, codes, sb, N, H, flags=0, ws=None):
    """One call through the C ABI; returns y (bf16, cpu), y_f32 (float64),
    the live count and the live index list (ascending, count entries)."""
    if ws is None:
        ws = torch.zeros(hs.hs_expert_down_sparse_workspace_size(N, H), dtype=torch.uint8, device="cuda")
    y = torch.empty(H, dtype=torch.bfloat16, device="cuda")
    yf = torch.empty(H, dtype=torch.float32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    idx = torch.full((N + 1,), -7, dtype=torch.int32, device="cuda")
    hs.hs_expert_down_sparse(h.cuda().float().contiguous(), codes, sb, N, H, y, yf, cnt, flags, ws, live_idx=idx)
    torch.cuda.synchronize()
    assert hs.hs_device_status() == hs.HS_OK
    c = int(cnt.item())
    li = idx.cpu().numpy()
    assert (li[c:] == -7).all(), "live_idx written past the live count"
    return y.cpu(), yf.cpu().double().numpy(), c, li[:c]


def check_live_idx(li, h, dense=False):
    """The kernel's rows read equal the oracle's live set {n : h_n > 0}
    (h is given, so the set is exact), ascending; every row when dense."""
    h = np.asarray(h, dtype=np.float64)
    want = np.arange(len(h)) if dense else np.asarray(oracle.live_set(h))
    assert np.array_equal(li, want), (len(li), len(want))


@pytest.mark.parametrize("H,N", [(64, 64), (128, 192), (256, 320), (2688, 1856), (2688, 3712), (3072, 128)])
def test_repack_matches_oracle_dequant(H, N):
    down = synth.gen_proj(H, N, (0, "repack", H, N))
    codes, sb = repack(down)
    w_nm = dequant_neuron_major(codes, sb)
    assert np.array_equal(w_nm, oracle.dequant(down))


def test_single_expert_down_parity():
    """Routed expert 2688x1856, h = relu(z)^2 with about 10% live."""
    h, down = synth.single_expert_down(0)
    codes, sb = repack(down)
    y, yf, cnt, li = run_down(h, codes, sb, 1856, 2688)
    ref = oracle.down_dense(h, down)
    check_close(yf, ref, "single expert y_f32")
    check_bf16_within_one_ulp(y, ref, "single expert y_bf16", yf)
    check_live_idx(li, h.double().numpy())  # live set exact: h is given


def test_twelve_neuron_golden_bit_exact():
    """The hand-worked 12-neuron example; every value is dyadic, so fp32 is exact."""
    rows = {}
    with open(os.path.join(GOLD, "relu2_12.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                k, *v = line.split()
                rows[k] = [float(t) for t in v]
    h = np.zeros(64)
    h[:12] = rows["h"]
    H = 64
    q = np.array([[(n + 3 * o) % 16 for n in range(64)] for o in range(H)], dtype=np.uint8)
    codes_om = torch.from_numpy((q[:, 0::2] | (q[:, 1::2] << 4)).astype(np.uint8))
    down = synth.W4Proj(codes_om, torch.ones((H, 1), dtype=torch.float16), torch.full((H, 1), -8.0, dtype=torch.float16))
    codes, sb = repack(down)
    y, yf, cnt, li = run_down(torch.from_numpy(h).float(), codes, sb, 64, H)
    assert yf[:4].tolist() == rows["y"]
    assert li.tolist() == [int(v) for v in rows["live"]]
    assert np.array_equal(yf, oracle.down_dense(h, down))


def test_dense_flag_equals_sparse_and_is_deterministic():
    h, down = synth.single_expert_down(0)
    codes, sb = repack(down)
    ws = torch.zeros(hs.hs_expert_down_sparse_workspace_size(1856, 2688), dtype=torch.uint8, device="cuda")
    y1, yf1, c1, l1 = run_down(h, codes, sb, 1856, 2688, ws=ws)
    y2, yf2, c2, l2 = run_down(h, codes, sb, 1856, 2688, ws=ws)   # same workspace: counters back at zero
    yd, yfd, cd, ld = run_down(h, codes, sb, 1856, 2688, flags=hs.HS_FORCE_DENSE, ws=ws)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2) and np.array_equal(l1, l2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    check_live_idx(ld, h.double().numpy(), dense=True)
    assert cd == 1856


@pytest.mark.parametrize("case", ["all_dead", "one_live_last_group", "all_live", "neg_zero_and_tiny", "group_dead"])
def test_edge_cases(case):
    N, H = 256, 2688
    down = synth.gen_proj(H, N, (0, "edge", case))
    codes, sb = repack(down)
    rng = np.random.default_rng(5)
    h = np.zeros(N, dtype=np.float32)
    if case == "one_live_last_group":
        h[N - 1] = 1.75
    elif case == "all_live":
        h[:] = rng.uniform(0.01, 2.0, N)
    elif case == "neg_zero_and_tiny":
        h[:] = -0.0
        h[3] = 1e-30
        h[100] = np.float32(2.0 ** -126)
        h[200] = 3.0
    elif case == "group_dead":
        h[:] = rng.uniform(0.01, 2.0, N)
        h[64:128] = 0.0
    y, yf, cnt, li = run_down(torch.from_numpy(h), codes, sb, N, H)
    ref = oracle.down_dense(h.astype(np.float64), down)
    check_live_idx(li, h)
    if case == "all_dead":
        assert np.all(yf == 0) and torch.all(y.float() == 0)
    else:
        check_close(yf, ref, case)
        check_bf16_within_one_ulp(y, ref, case, yf)


@pytest.mark.parametrize("H,N", [(64, 64), (64, 128), (128, 192), (512, 64), (3072, 320), (128, 4096), (128, 4160),
                                 (192, 8192)])
def test_small_shapes_vs_oracle(H, N):
    """Small and wide experts (up to 128 groups of 64 neurons)."""
    down = synth.gen_proj(H, N, (1, "small", H, N))
    codes, sb = repack(down)
    rng = np.random.default_rng(H + N)
    z = rng.normal(-0.8, 1.0, N)
    h = oracle.relu2(z).astype(np.float32)
    y, yf, cnt, li = run_down(torch.from_numpy(h), codes, sb, N, H)
    ref = oracle.down_dense(h.astype(np.float64), down)
    check_close(yf, ref, f"{H}x{N}")
    check_bf16_within_one_ulp(y, ref, f"{H}x{N}", yf)
    check_live_idx(li, h)


@pytest.mark.parametrize("N", [4096, 4160])
def test_dense_flag_equals_sparse_wide_experts(N):
    """HS_FORCE_DENSE gives the sparse result bit for bit for wide experts
    too, and repeats are identical."""
    H = 256
    down = synth.gen_proj(H, N, (2, "both", N))
    codes, sb = repack(down)
    z = np.random.default_rng(N).normal(-1.2815516, 1.0, N)
    h = torch.from_numpy(oracle.relu2(z).astype(np.float32))
    y1, yf1, c1, l1 = run_down(h, codes, sb, N, H)
    y2, yf2, c2, l2 = run_down(h, codes, sb, N, H)
    yd, yfd, cd, ld = run_down(h, codes, sb, N, H, flags=hs.HS_FORCE_DENSE)
    assert np.array_equal(yf1, yf2) and torch.equal(y1, y2) and np.array_equal(l1, l2)
    assert np.array_equal(yf1, yfd) and torch.equal(y1, yd)
    check_live_idx(l1, h.numpy())
    assert cd == N


def test_one_workspace_across_shapes_and_repeats():
    """Every call leaves the workspace's completion counters at zero, so one
    zero-filled workspace (sized for the largest shape) serves a sequence of
    calls of different shapes and band counts, each equal to a call on a
    fresh workspace."""
    shapes = [(2688, 1856), (64, 64), (3072, 4096), (256, 320), (2688, 1856)]
    big = max(hs.hs_expert_down_sparse_workspace_size(N, H) for H, N in shapes)
    ws = torch.zeros(big, dtype=torch.uint8, device="cuda")
    for i, (H, N) in enumerate(shapes):
        down = synth.gen_proj(H, N, (3, "reuse", H, N))
        codes, sb = repack(down)
        z = np.random.default_rng(i).normal(-1.2815516, 1.0, N)
        h = torch.from_numpy(oracle.relu2(z).astype(np.float32))
        y, yf, c, li = run_down(h, codes, sb, N, H, ws=ws)
        y0, yf0, c0, l0 = run_down(h, codes, sb, N, H)
        assert np.array_equal(yf, yf0) and torch.equal(y, y0) and np.array_equal(li, l0)
        check_live_idx(li, h.numpy())
        check_close(yf, oracle.down_dense(h.double().numpy(), down), f"reuse {H}x{N}")
