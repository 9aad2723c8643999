"""The prefill row gather's planner (hs_rowgather.cuh), on the CPU.

"Skipping dead neurons..." section "What we do instead": per token tile, the
neurons live for some token of the tile are gathered into a dense product.
The planner packs each tile's union-live neurons into 64-entry k-steps.  Its
header is host-compilable: the C++ driver built here checks every plan's
invariants on random and adversarial masks, and the planner's k-step counts
are compared with the rule restated in tests/_util.plan_ksteps, which the GPU
tests use to predict the kernel's skip counts from its own live masks.
"""
import pathlib
import shutil
import subprocess

import numpy as np
import pytest

from _util import plan_ksteps

ROOT = pathlib.Path(__file__).resolve().parents[1]


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ is not available")
    exe = tmp_path_factory.mktemp("rg") / "rowgather_plan_check"
    subprocess.run([cxx, "-O2", "-std=c++17", "-I", str(ROOT / "activation_sparse_moe_gb300" / "csrc"),
                    str(ROOT / "tests" / "rowgather_plan_check.cpp"), "-o", str(exe)], check=True)
    return exe


def test_planner_invariants(checker):
    r = subprocess.run([str(checker)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stderr


def _masks(rng, NG, q, clustered=0):
    bits = rng.random((NG, 64)) < q
    for g in rng.choice(NG, size=min(clustered, NG), replace=False):
        bits[g] = False
    return [sum(1 << int(i) for i in np.flatnonzero(row)) for row in bits]


def test_restated_rule_matches_planner(checker):
    rng = np.random.default_rng(0)
    cases = []
    for NG in (1, 2, 3, 29, 58, 64):
        for q in (0.0, 0.01, 0.05, 0.1, 0.3, 0.7, 0.95, 1.0):
            for clustered in (0, NG // 3):
                for _ in range(6):
                    cases.append(_masks(rng, NG, q, clustered))
    # hand cases: 8 live + dead + full (2 k-steps); alternating 8 and 64; one neuron per group
    cases += [[0xFF, 0, (1 << 64) - 1], [0xFF, (1 << 64) - 1] * 8, [1] * 29, [(1 << 9) - 1] * 58]
    text = "".join(f"{len(m)} " + " ".join(f"{w:x}" for w in m) + "\n" for m in cases)
    r = subprocess.run([str(checker), "plan"], input=text, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    got = [tuple(map(int, line.split())) for line in r.stdout.split("\n") if line]
    assert len(got) == len(cases)
    for m, (n, ident) in zip(cases, got):
        assert plan_ksteps(m) == n, (len(m), [hex(w) for w in m][:4], n, ident)
    # closed forms: all dead -> 0 k-steps; all live -> NG; one live neuron in each of NG groups -> ceil(NG / 2)
    assert plan_ksteps([0] * 29) == 0 and plan_ksteps([(1 << 64) - 1] * 29) == 29
    assert plan_ksteps([1] * 29) == 15
