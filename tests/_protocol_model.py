"""An interleaving model of the mbarrier protocols of the tensor-core kernels.

Each warp role of a kernel is a generator that performs the role's arrivals
(TMA completion, tcgen05.commit, mbarrier.arrive) and yields the waits it makes,
in the order of the kernel's code.  A barrier completes a phase when its
arrivals reach its count; a wait on parity P succeeds once the phase of parity
P has completed, i.e. while the barrier's current phase parity differs from P
(so a fresh barrier lets parity 1 pass at once, the convention the kernels use
for "buffer initially free").  Asynchronous operations complete at once in the
model: one legal schedule among many; the random interleaving of the roles
explores the others.  Roles also assert the buffer hazards the barriers exist
to prevent (a buffer refilled while still being read).
"""
from __future__ import annotations

import random
from typing import Dict, Iterator, List, Optional, Tuple


class Bar:
    def __init__(self, count: int):
        self.count, self.arrivals, self.done = count, 0, 0

    def arrive(self) -> None:
        self.arrivals += 1
        if self.arrivals == self.count:
            self.arrivals, self.done = 0, self.done + 1

    def passed(self, parity: int) -> bool:
        return (self.done & 1) != parity


Wait = Tuple[Bar, int]


def run(roles: List[Iterator[Optional[Wait]]], seed: int, max_steps: int = 200000) -> bool:
    """Interleave the roles at random until all finish (True) or none can move (False)."""
    rng = random.Random(seed)
    live: Dict[int, Iterator] = dict(enumerate(roles))
    pending: Dict[int, Optional[Wait]] = {i: None for i in live}
    for _ in range(max_steps):
        if not live:
            return True
        ready = [i for i in live if pending[i] is None or pending[i][0].passed(pending[i][1])]
        if not ready:
            return False
        i = rng.choice(ready)
        try:
            pending[i] = next(live[i])
        except StopIteration:
            del live[i]
    return False


def named_barrier(bar: Bar, use: int):
    """The use-th bar.sync among bar.count roles: arrive, then wait for that phase."""
    bar.arrive()
    yield (bar, use & 1)


# ---------------------------------------------------------------------------
# indexer_kernel: TMA producer -> stage ring -> MMA -> two TMEM accumulators ->
# two epilogue groups of four warps alternating tiles (one item per CTA)

def indexer(ntile: int, stages: int, seed: int) -> bool:
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(1) for _ in range(stages)]
    tfull, tempty = [Bar(1), Bar(1)], [Bar(4), Bar(4)]
    qfull = Bar(1)
    loads = [0] * stages

    def producer():
        qfull.arrive()
        for i in range(ntile):
            s, ph = i % stages, (i // stages) & 1
            yield (empty[s], ph ^ 1)
            assert empty[s].done >= i // stages, "stage refilled before its MMAs read it"
            loads[s] += 1
            full[s].arrive()

    def mma():
        yield (qfull, 0)
        for i in range(ntile):
            s, ph = i % stages, (i // stages) & 1
            acc, aph = i & 1, (i >> 1) & 1
            yield (tempty[acc], aph ^ 1)
            yield (full[s], ph)
            assert loads[s] == i // stages + 1, "MMA read a stage that holds another tile"
            assert tempty[acc].done >= i >> 1, "accumulator overwritten before the epilogue read it"
            empty[s].arrive()
            tfull[acc].arrive()

    def epilogue(group: int):
        for i in range(group, ntile, 2):
            acc, aph = i & 1, (i >> 1) & 1
            yield (tfull[acc], aph)
            tempty[acc].arrive()

    return run([producer(), mma()] + [epilogue(g) for g in (0, 1) for _ in range(4)], seed)


# ---------------------------------------------------------------------------
# attend_tc_kernel: K tiles loaded at once, a tile's buffer refilled with V
# once its score MMAs are done (gather or TMA producers alike), per-tile
# epilogue (two named barriers per tile among the 8 epilogue warps), output
# MMAs after every tile's P rows and V rows, one final commit

def attend_tc(ntile: int, seed: int) -> bool:
    q = Bar(1)
    kfull = [Bar(1) for _ in range(ntile)]
    vfull = [Bar(1) for _ in range(ntile)]
    sdone = [Bar(1) for _ in range(ntile)]
    pfull = [Bar(8) for _ in range(ntile)]
    ofull = Bar(1)
    epi_bar = Bar(8)
    buffer = ["empty"] * ntile

    def producer():
        q.arrive()
        for j in range(ntile):
            buffer[j] = "K"
            kfull[j].arrive()
        for j in range(ntile):
            yield (sdone[j], 0)
            assert sdone[j].done >= 1, "V loaded over K rows still being read"
            buffer[j] = "V"
            vfull[j].arrive()

    def mma():
        yield (q, 0)
        for j in range(ntile):
            yield (kfull[j], 0)
            assert buffer[j] == "K"
            sdone[j].arrive()
        for j in range(ntile):
            yield (pfull[j], 0)
            yield (vfull[j], 0)
            assert buffer[j] == "V"
        ofull.arrive()

    def epilogue(me: int):
        for j in range(ntile):
            yield (sdone[j], 0)
            yield from named_barrier(epi_bar, 2 * j)      # the quarters' maxima
            yield from named_barrier(epi_bar, 2 * j + 1)  # the per-head offsets
            pfull[j].arrive()
        yield from named_barrier(epi_bar, 2 * ntile)      # the sums
        yield from named_barrier(epi_bar, 2 * ntile + 1)  # the coefficients
        yield (ofull, 0)

    return run([producer(), mma()] + [epilogue(w) for w in range(8)], seed)
