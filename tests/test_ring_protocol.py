"""The prefill GEMMs' mbarrier rings, modelled on the CPU.

Both tensor-core products of the prefill run a warp-specialised pipeline:
one producer loads the 4-bit codes into a weight ring, another the 16-bit
operand into a stage ring, four dequantising groups take the k-steps round
robin (step q goes to group q % 4) and one thread issues the MMAs, whose
commits release the stages in order.  Every wait is a parity test on an
mbarrier, which is sound only while the barrier is at most one phase behind
the phase waited for: two phases behind, the incomplete phase has the parity
of the one wanted and the test passes at once.

This model runs that protocol under random schedules, with copies that land
out of order (as TMA copies may) and in-order commits, and records every
wait that passed on such an aliased parity, every read of a slot whose copy
had not landed, and every arrival on a barrier phase that had none left.
The ring depths and the order of the dequantisers' two waits are read from
the kernel source, so the test follows the committed code; the model is
also shown to catch the fault on a configuration that has it (a weight ring
of depth 5 waited on before the stage release).
"""
import pathlib
import random
import re

import pytest

SRC = pathlib.Path(__file__).resolve().parents[1] / "activation_sparse_moe_gb300" / "csrc" / "hs_prefill.cu"
GROUPS = 4


def committed_rings():
    """(WD, SD, stage-release-first) of the up and down kernels, from the source."""
    s = SRC.read_text()
    up = re.search(r"constexpr int kUpWD = (\d+), kUpSD = (\d+);", s)
    dn = re.search(r"constexpr int kDnWD = (\d+), kDnSD = (\d+);", s)
    assert up and dn
    # the dequantisers' combined wait names the stage ring first when it waits for the release first
    up_first = bool(re.search(r"__all_sync\(0xffffffffu, wait_free\(br\.sempty, kUpSD, qk\) && wait_full\(br\.wfull",
                              s))
    dn_first = bool(re.search(r"__all_sync\(0xffffffffu, wait_free\(br\.sempty, kDnSD, qk\) && wait_full\(br\.wfull",
                              s))
    assert re.search(r"wait_full\(br\.wfull, kUpWD, qk\)", s) and re.search(r"wait_full\(br\.wfull, kDnWD, qk\)", s)
    return {"up": (int(up[1]), int(up[2]), up_first), "down": (int(dn[1]), int(dn[2]), dn_first)}


class Barrier:
    """An mbarrier: expected arrivals per phase, pending arrivals and bytes, completed phases."""

    def __init__(self, count, faults):
        self.count, self.pending, self.tx, self.done = count, count, 0, 0
        self.faults = faults

    def arrive(self, tx=0):
        if self.pending == 0:
            self.faults.append("arrival on a phase with no arrival left")
        self.pending -= 1
        self.tx += tx
        self._maybe_complete()

    def land(self, tx):
        self.tx -= tx
        self._maybe_complete()

    def _maybe_complete(self):
        if self.pending <= 0 and self.tx == 0:
            self.done += 1
            self.pending, self.tx = self.count, 0

    def parity_full(self, use):
        """try_wait.parity for use `use` complete; (passes, sound)."""
        passes = (self.done & 1) != (use & 1)
        return passes, self.done >= use + 1

    def parity_free(self, use):
        """The producer-side form: the slot's use `use - 1` released."""
        passes = (self.done & 1) == (use & 1)
        return passes, self.done >= use


def run_pipeline(WD, SD, release_first, steps, seed):
    """One schedule of the pipeline; returns the list of faults seen."""
    rng = random.Random(seed)
    faults = []
    wfull = [Barrier(1, faults) for _ in range(WD)]
    wempty = [Barrier(1, faults) for _ in range(WD)]     # one arrival per group (its warps as one)
    sfull = [Barrier(2, faults) for _ in range(SD)]      # the stage copy + the group's arrival
    sempty = [Barrier(1, faults) for _ in range(SD)]     # the MMA commit
    landed = [-1] * WD                                   # k-step whose codes sit in each weight slot
    events = []                                          # (time, seq, action)
    seq = [0]

    def later(t, fn):
        seq[0] += 1
        events.append((t, seq[0], fn))

    # gw: how many of its two waits the group has passed for its current k-step
    # (a wait loops until it passes; a passed wait is not tested again)
    state = {"wq": 0, "xq": 0, "mq": 0, "gq": [g for g in range(GROUPS)], "gw": [0] * GROUPS, "last_commit": 0}

    def try_wait(bar, use, kind):
        ok, sound = (bar.parity_full(use) if kind == "full" else bar.parity_free(use))
        if ok and not sound:
            faults.append(f"{kind} wait passed on an aliased parity")
        return ok

    def step_w(t):
        q = state["wq"]
        if q >= steps or not try_wait(wempty[q % WD], q // WD, "free"):
            return
        s = q % WD
        wfull[s].arrive(tx=1)

        def land(q=q, s=s):
            landed[s] = q
            wfull[s].land(1)
        later(t + rng.choice([1, 2, 3, 5, 8, 40]), land)
        state["wq"] += 1

    def step_x(t):
        q = state["xq"]
        if q >= steps or not try_wait(sempty[q % SD], q // SD, "free"):
            return
        s = q % SD
        sfull[s].arrive(tx=1)
        later(t + rng.choice([1, 2, 3, 5, 8, 40]), lambda s=s: sfull[s].land(1))
        state["xq"] += 1

    def step_g(t, g):
        q = state["gq"][g]
        if q >= steps:
            return
        waits = [(sempty[q % SD], q // SD, "free"), (wfull[q % WD], q // WD, "full")]
        if not release_first:
            waits.reverse()
        # the combined wait: the first test must pass before the second is tried
        while state["gw"][g] < 2:
            bar, use, kind = waits[state["gw"][g]]
            if not try_wait(bar, use, kind):
                return
            state["gw"][g] += 1
        state["gw"][g] = 0
        if landed[q % WD] != q:
            faults.append(f"k-step {q} read a weight slot holding k-step {landed[q % WD]}")
        sfull[q % SD].arrive()
        wempty[q % WD].arrive()
        state["gq"][g] += GROUPS

    def step_mma(t):
        q = state["mq"]
        if q >= steps or not try_wait(sfull[q % SD], q // SD, "full"):
            return
        done = max(state["last_commit"], t) + rng.choice([1, 2, 4, 12])
        state["last_commit"] = done
        later(done, lambda s=q % SD: sempty[s].arrive())
        state["mq"] += 1

    actors = [step_w, step_x, step_mma] + [lambda t, g=g: step_g(t, g) for g in range(GROUPS)]
    t = 0
    while state["mq"] < steps or events:
        due = sorted(e for e in events if e[0] <= t)
        for e in due:
            events.remove(e)
            e[2]()
        order = list(range(len(actors)))
        rng.shuffle(order)
        for i in order:
            if rng.random() < 0.6:
                actors[i](t)
        t += 1
        if t > 200 * steps:
            faults.append("no progress")
            break
    return faults


@pytest.mark.parametrize("kernel", ["up", "down"])
def test_committed_rings_never_alias(kernel):
    WD, SD, first = committed_rings()[kernel]
    for seed in range(60):
        faults = run_pipeline(WD, SD, first, steps=96, seed=seed)
        assert not faults, (kernel, WD, SD, first, seed, faults[:3])


def test_model_catches_the_aliasing_ring():
    """A weight ring of depth 5 under four groups, waited on before the stage
    release: some schedule passes a wait on an aliased parity and reads codes
    that have not landed."""
    seen = []
    for seed in range(200):
        seen += run_pipeline(5, 4, False, steps=96, seed=seed)
        if any("aliased" in f for f in seen) and any("read a weight slot" in f for f in seen):
            break
    assert any("aliased" in f for f in seen)
    assert any("read a weight slot" in f for f in seen)


def test_model_catches_a_six_deep_stage_ring():
    """Depth 6 for both rings (not a multiple of the group count) with the
    weight wait first: the model finds the fault there too."""
    seen = []
    for seed in range(200):
        seen += run_pipeline(6, 6, False, steps=96, seed=seed)
        if seen:
            break
    assert seen
