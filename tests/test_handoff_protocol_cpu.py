"""A CPU model of the prefill kernel's handoffs between a query tile's MMA
warp and its softmax warpgroup, run under random interleavings, random MMA
completion times and random aborts (bounded waits that run out).

The kernel (tiled attention forward, the cruxr.ai "FlashAttention" inner loop
over K/V blocks) passes each K/V block of a query tile through two named
barriers: "S read" (separate-P layout, d = 64) and "P written".  The four
softmax warps only arrive at them; the MMA warp syncs.  The MMA warp signals
"S full" and "P V done" on mbarriers (tcgen05.commit, or a plain arrival
after an abort).  A named barrier completes when 160 threads have arrived,
whatever phase they meant; an mbarrier wait is a parity wait.  The model
checks, for every schedule it draws, that

  * every role finishes (no barrier is left waiting), and
  * every completed named-barrier phase holds the arrivals of one K/V block
    only (an arrive-only side running a phase ahead would mix blocks).

It also runs the protocol as it was before the abort path kept the signals
and their waits, and checks that the model finds the hang there: the
softmax warps, skipping their waits after an abort, arrive ahead.  The
kernel's side of this is in attn_fwd_sm103.cuh: the MMA warp's plain
arrivals on S full and P V done after an abort, and the softmax's
mbar_wait_signal waits."""
import random

import pytest

SOFTMAX_WARPS = 4
WARP = 32
HANDOFF_THREADS = SOFTMAX_WARPS * WARP + WARP


class NamedBarrier:
    def __init__(self, name):
        self.name = name
        self.count = 0
        self.tags = []
        self.phase = 0
        self.mixed = []

    def arrive(self, tag):
        self.count += WARP
        self.tags.append(tag)
        if self.count >= HANDOFF_THREADS:
            assert self.count == HANDOFF_THREADS
            if len(set(self.tags)) != 1:
                self.mixed.append((self.name, list(self.tags)))
            self.count = 0
            self.tags = []
            self.phase += 1
            return self.phase - 1  # the phase this arrival completed
        return self.phase


class MBarrier:
    """Count-1 mbarrier: each arrival completes a phase."""

    def __init__(self):
        self.completed = 0

    def arrive(self):
        self.completed += 1

    def try_wait_parity(self, parity):
        return (self.completed & 1) != parity


class Kernel:
    def __init__(self, rng, items, separate_p, p_fail, fixed):
        self.rng = rng
        self.items = items  # K/V blocks of each item
        self.sep = separate_p
        self.p_fail = p_fail  # chance that a pending bounded wait runs out at a step
        self.fixed = fixed
        self.abort = False
        self.bar_p = NamedBarrier("P")
        self.bar_sread = NamedBarrier("SRead")
        self.s_full = MBarrier()
        self.pv_done = MBarrier()
        self.o_final = MBarrier()
        self.pending = []  # tensor-core commits in flight: callables

    # a bounded wait in the normal mode: True once the barrier phase is seen;
    # False when the wait runs out or sees the abort flag
    def wait_ok(self, bar, parity):
        while True:
            if bar.try_wait_parity(parity):
                return True
            if self.abort and self.rng.random() < 0.5:
                return False
            if self.rng.random() < self.p_fail:
                self.abort = True
                return False
            yield "wait"

    def drain(self, bar, parity):
        while not bar.try_wait_parity(parity):
            yield "drain"

    def sync(self, nb, tag):
        ph = nb.arrive(tag)
        while nb.phase <= ph:
            yield "sync"

    def mma_warp(self):
        ok = True
        pending = None  # (tag,) of the P V to issue

        def issue_qk(tag):
            nonlocal ok
            if ok:
                self.pending.append(self.s_full.arrive)
            elif self.fixed:
                self.s_full.arrive()

        def issue_pv(tag, last):
            nonlocal ok
            yield from self.sync(self.bar_p, tag)
            ok = ok and not self.abort
            if not ok and self.fixed:
                if self.sep:
                    self.pv_done.arrive()
                if last:
                    self.o_final.arrive()
            if ok:
                def commit():  # P V done and, for an item's last block, O final: one MMA completion
                    if self.sep:
                        self.pv_done.arrive()
                    if last:
                        self.o_final.arrive()
                self.pending.append(commit)

        for it, n in enumerate(self.items):
            for j in range(n):
                tag = (it, j)
                if self.sep:
                    if j > 0:
                        yield from self.sync(self.bar_sread, (it, j - 1))
                    if ok:  # K/V tile wait
                        ok = yield from self.maybe_fail()
                    issue_qk(tag)
                    if pending is not None:
                        yield from issue_pv(pending, False)
                else:
                    if pending is not None:
                        yield from issue_pv(pending, False)
                    if ok:
                        ok = yield from self.maybe_fail()
                    issue_qk(tag)
                pending = tag
            if self.sep:
                yield from self.sync(self.bar_sread, (it, n - 1))
            yield from issue_pv(pending, True)
            pending = None

    def maybe_fail(self):
        # a wait on a producer barrier: succeeds, or runs out / sees the abort
        if self.abort and self.rng.random() < 0.5:
            return False
        if self.rng.random() < self.p_fail:
            self.abort = True
            return False
        yield "kv"
        return True

    def softmax_warp(self):
        """One softmax warp, following the kernel's loop.  With the fix, the
        S-full and P V-done waits do not poll the abort flag (the MMA warp
        signals them in every case) and the block's work always runs, so the
        warp arrives at S-read and P only after the signal that follows the
        MMA warp's sync of the previous phase.  Without it (the old
        protocol), a failed wait skips the waits of every later block."""
        ok = True
        ns = npv = nfin = 0
        for it, n in enumerate(self.items):
            for j in range(n):
                if self.fixed:
                    yield from self.drain(self.s_full, ns & 1)
                elif ok:
                    ok = yield from self.wait_ok(self.s_full, ns & 1)
                ns += 1
                if self.sep:
                    self.bar_sread.arrive((it, j))
                if self.fixed or ok:
                    yield "exp"
                    if self.sep and j > 0:
                        if self.fixed:
                            yield from self.drain(self.pv_done, (npv - 1) & 1)
                        else:
                            ok = (yield from self.wait_ok(self.pv_done, (npv - 1) & 1)) and ok
                self.bar_p.arrive((it, j))
                npv += 1
            # epilogue: O final (with the fix, also a signal wait; it covers
            # the item's last P V done, which no block waits for)
            if self.fixed:
                yield from self.drain(self.o_final, nfin & 1)
            elif ok:
                ok = yield from self.wait_ok(self.o_final, nfin & 1)
            nfin += 1
            yield "epilogue"

    def run(self, max_idle=4000):
        """'done', or 'hang' when no role has moved for max_idle steps with
        no tensor-core commit left to complete."""
        live = [self.mma_warp()] + [self.softmax_warp() for _ in range(SOFTMAX_WARPS)]
        idle = 0
        while live:
            if self.pending and self.rng.random() < 0.3:  # MMAs complete at random times
                self.pending.pop(0)()
                idle = 0
            a = self.rng.choice(live)
            try:
                state = next(a)
            except StopIteration:
                live.remove(a)
                idle = 0
                continue
            idle = idle + 1 if state in ("wait", "drain", "sync") else 0
            if idle > max_idle and not self.pending:
                return "hang"
        return "done"


def run_trials(fixed, trials, seed):
    rng = random.Random(seed)
    outcomes = {"done": 0, "hang": 0, "mixed": 0}
    for _ in range(trials):
        items = [rng.randint(1, 4) for _ in range(rng.randint(1, 3))]
        k = Kernel(rng, items, rng.random() < 0.5, rng.choice([0.0, 0.002, 0.02, 0.3, 0.9]), fixed)
        outcomes[k.run()] += 1
        if k.bar_p.mixed or k.bar_sread.mixed:
            outcomes["mixed"] += 1
    return outcomes


def test_no_hang_and_no_mixed_phase_under_aborts():
    out = run_trials(fixed=True, trials=3000, seed=7)
    assert out["hang"] == 0 and out["mixed"] == 0, out
    assert out["done"] == 3000


def test_model_finds_the_old_abort_path_hang():
    """Planted in the model only: the protocol without the abort-path signals
    hangs or mixes phases on some schedules."""
    out = run_trials(fixed=False, trials=3000, seed=7)
    assert out["hang"] + out["mixed"] > 0, out


@pytest.mark.parametrize("sep", [False, True])
def test_no_abort_runs_clean(sep):
    rng = random.Random(11)
    for _ in range(300):
        items = [rng.randint(1, 5) for _ in range(rng.randint(1, 4))]
        k = Kernel(rng, items, sep, 0.0, True)
        assert k.run() == "done" and not k.bar_p.mixed and not k.bar_sread.mixed
