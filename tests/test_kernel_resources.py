"""Register and spill budget of every kernel, from ptxas's report of the
build (CPU; nvcc cross-compiles for sm_103a without a GPU).

The hot kernels are sized for a fixed residency (two 256-thread CTAs per SM
for the batch-1 and batch decode kernels: at most 128 registers a thread),
and several sit close to that limit, where a small change of the code can
make the compiler spill registers on the main path (it did once, costing the
persistent batch kernel 13% at 32 tokens).  No kernel may spill, except the
instantiation of the persistent batch kernel that also writes the debug live
masks (used only when a caller asks for them).
"""
import pytest

from activation_sparse_moe_gb300 import build as hsbuild

DEBUG_ONLY = ("_ZN2hs18batch_fused_kernelILb1EEEvNS_11LayerParamsENS_7BatchIOE",)
# kernels launched with two 256-thread CTAs per SM (__launch_bounds__(256, 2))
TWO_PER_SM = ("moe_decode_b1_kernel", "batch_small_kernel", "batch_fused_kernel")


@pytest.fixture(scope="module")
def report():
    hsbuild.build()
    try:
        rep = hsbuild.resource_report()
    except FileNotFoundError:
        hsbuild.build(force=True)
        rep = hsbuild.resource_report()
    assert rep, "no ptxas report"
    return rep


def test_no_kernel_spills(report):
    spilling = {k: v for k, v in report.items()
                if (v["spill_stores"] or v["spill_loads"]) and k not in DEBUG_ONLY}
    assert not spilling, spilling


def test_two_cta_kernels_fit_their_register_budget(report):
    found = 0
    for name, v in report.items():
        if any(k in name for k in TWO_PER_SM):
            found += 1
            assert v["regs"] <= 128, (name, v)
    assert found >= 4

