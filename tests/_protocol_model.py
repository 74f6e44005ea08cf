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
# indexer_kernel (persistent): a CTA walks a list of items (query group x tile
# range; ntile may be 0 = nothing visible, skipped by every role).  Key
# producer -> stage ring -> MMA -> two TMEM accumulators -> two epilogue groups
# of four warps, both on every tile (each group half of the item's queries:
# eight arrivals free an accumulator); an item producer fills the
# double-buffered head weights (wfull / wfree) and the single query buffer
# (qfull, refilled once the MMAs of the previous item are done: qfree); with
# the histogram both groups meet at every item's end (two named barriers).

def indexer(items, stages: int, seed: int, hist: bool = False, plant: str = "", fp8: bool = False,
            groups=None, epi_groups: int = 2) -> bool:
    """``items``: tile counts of the CTA's items in order (0 = nothing
    visible, skipped); ``groups``: the query group of each item (consecutive
    items of one group share the query rows, loaded once, and the histogram,
    flushed once).  ``plant`` names a wait to leave out ("qfree", "wfree",
    "sfree"), for the tests that show the hazard checks catch a missing wait.
    ``fp8``: the key scales share the stage ring and a stage's scale slot is
    released by the epilogue warps that read it (sfree).  ``epi_groups``:
    epilogue groups of four warps (two, or four when H_I <= 64), all on
    every tile."""
    nw = 4 * epi_groups
    groups = list(range(len(items))) if groups is None else groups
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(1) for _ in range(stages)]
    sfree = [Bar(nw) for _ in range(stages)]
    scale_tile = [-1] * stages    # the tile whose key scales each stage's slot holds
    tfull, tempty = [Bar(1), Bar(1)], [Bar(nw), Bar(nw)]
    qfull, qfree = Bar(1), Bar(1)
    wfull, wfree = [Bar(1), Bar(1)], [Bar(epi_groups), Bar(epi_groups)]
    group_bar = [Bar(4) for _ in range(epi_groups)]
    epi_bar = Bar(nw)
    live = [(n, g) for n, g in zip(items, groups) if n > 0]
    loads = [0] * stages
    q_group = [None]              # the query group whose rows the buffer holds
    w_item = [-1, -1]             # the item whose weights each buffer holds
    mma_groups_done = [0]         # query groups whose MMAs have completed
    epi_done = [[0] * epi_groups, [0] * epi_groups]  # [buffer][group]: items of that parity finished by the group

    def new_group(it):
        return it == 0 or live[it][1] != live[it - 1][1]

    def key_producer():
        gt = 0
        for n in items:
            for _ in range(max(n, 0)):
                s, ph = gt % stages, (gt // stages) & 1
                yield (empty[s], ph ^ 1)
                assert empty[s].done >= gt // stages, "stage refilled before its MMAs read it"
                if fp8 and plant != "sfree":
                    yield (sfree[s], ph ^ 1)
                if fp8:
                    assert gt < stages or sfree[s].done >= gt // stages, "key scales refilled before the epilogue read them"
                    scale_tile[s] = gt
                loads[s] += 1
                full[s].arrive()
                gt += 1

    def item_producer():
        # per item: the query rows when its group is new (the MMAs wait for
        # them), then the weights
        nq = 0
        for it in range(len(live)):
            ib = it & 1
            if new_group(it):
                if nq >= 1 and plant != "qfree":
                    yield (qfree, (nq - 1) & 1)
                    assert mma_groups_done[0] >= nq, "query rows refilled before the previous group's MMAs ended"
                q_group[0] = live[it][1]
                yield None
                qfull.arrive()
                nq += 1
            if it >= 2 and plant != "wfree":
                yield (wfree[ib], ((it - 2) >> 1) & 1)
                assert min(epi_done[ib]) >= (it - 2) // 2 + 1, "weights refilled while a group still reads them"
            w_item[ib] = it
            yield None
            wfull[ib].arrive()

    def mma():
        gt = nq = 0
        for it, (n, g) in enumerate(live):
            if new_group(it):
                if nq > 0:
                    mma_groups_done[0] += 1    # the commit completes once the previous group's MMAs are done
                    qfree.arrive()
                yield (qfull, nq & 1)
                nq += 1
            for _ in range(n):
                s, ph = gt % stages, (gt // stages) & 1
                acc, aph = gt & 1, (gt >> 1) & 1
                yield (tempty[acc], aph ^ 1)
                yield (full[s], ph)
                assert loads[s] == gt // stages + 1, "MMA read a stage that holds another tile"
                assert tempty[acc].done >= gt >> 1, "accumulator overwritten before the epilogue read it"
                assert q_group[0] == g, "MMA read another group's query rows"
                empty[s].arrive()
                tfull[acc].arrive()
                gt += 1

    def epilogue(group: int, first: bool):
        gt = 0
        uses = 0
        for it, (n, g) in enumerate(live):
            ib = it & 1
            yield (wfull[ib], (it >> 1) & 1)
            assert w_item[ib] == it, "epilogue read another item's weights"
            for i in range(n):
                g2 = gt + i
                acc = g2 & 1
                yield (tfull[acc], (g2 >> 1) & 1)
                assert tfull[acc].done >= (g2 >> 1) + 1 and tempty[acc].done == g2 >> 1, \
                    "epilogue read an accumulator another tile owns"
                if fp8:
                    st = g2 % stages
                    yield (full[st], (g2 // stages) & 1)
                    assert scale_tile[st] == g2, "epilogue read another tile's key scales"
                    sfree[st].arrive()
                tempty[acc].arrive()
            gt += n
            yield from named_barrier(group_bar[group], it)
            if first:
                epi_done[ib][group] += 1
                wfree[ib].arrive()
            if hist and (it + 1 == len(live) or live[it + 1][1] != g):
                yield from named_barrier(epi_bar, uses)
                yield from named_barrier(epi_bar, uses + 1)
                uses += 2

    roles = [key_producer(), item_producer(), mma()]
    roles += [epilogue(g, w == 0) for g in range(epi_groups) for w in range(4)]
    return run(roles, seed)


# ---------------------------------------------------------------------------
# indexer_single_kernel: one item per CTA -- thread 0 requests the query rows
# and the first min(stages, cap) key tiles before the visibility is known
# (cap: the item's tiles before the visibility cut; every stage is free then),
# the producer keeps the ring filled up to the ntile visible tiles, the MMA
# issuer feeds n_acc TMEM accumulators (2 or 4: tile i goes to i mod n_acc),
# two epilogue groups of four warps alternate tiles (group g reads the
# accumulators of the tiles i = g mod 2); with FP8 keys each stage's scale slot is released by the
# group that read it.  Every issued copy lands before the CTA exits, read or
# not (a pre-issued tile past the visible range is never read).

def indexer_single(ntile: int, stages: int, seed: int, fp8: bool = False, cap: Optional[int] = None,
                   n_acc: int = 2, plant: Optional[str] = None) -> bool:
    cap = ntile if cap is None else cap
    assert 0 <= ntile <= cap and n_acc in (2, 4)
    full = [Bar(1) for _ in range(stages)]
    empty = [Bar(1) for _ in range(stages)]
    sfree = [Bar(4) for _ in range(stages)]
    tfull, tempty = [Bar(1) for _ in range(n_acc)], [Bar(4) for _ in range(n_acc)]
    acc_tile = [-1] * n_acc
    qfull = Bar(1)
    loads = [0] * stages
    scale_tile = [-1] * stages
    n_pre = min(stages, cap)

    def load(i: int):
        s = i % stages
        if fp8:
            scale_tile[s] = i
        loads[s] += 1
        full[s].arrive()

    def producer():
        qfull.arrive()
        for i in range(n_pre):       # before the role split: no wait, every stage free
            load(i)
        issued = n_pre
        if ntile > 0:
            for i in range(n_pre, ntile):
                s, ph = i % stages, (i // stages) & 1
                yield (empty[s], ph ^ 1)
                assert empty[s].done >= i // stages, "stage refilled before its MMAs read it"
                if fp8:
                    yield (sfree[s], ph ^ 1)
                    assert sfree[s].done >= i // stages, "key scales refilled before the epilogue read them"
                load(i)
                issued = i + 1
        # drain: the last copy issued into each stage has landed
        for s in range(min(stages, issued)):
            last = issued - 1 - ((issued - 1 - s) % stages)
            yield (full[s], (last // stages) & 1)
        yield (qfull, 0)

    def mma():
        yield (qfull, 0)
        for i in range(ntile):
            s, ph = i % stages, (i // stages) & 1
            acc, aph = i % n_acc, (i // n_acc) & 1
            yield (tempty[acc], aph ^ 1)
            yield (full[s], ph)
            assert loads[s] == i // stages + 1, "MMA read a stage that holds another tile"
            assert tempty[acc].done >= i // n_acc, "accumulator overwritten before the epilogue read it"
            acc_tile[acc] = i
            empty[s].arrive()
            tfull[acc].arrive()

    def epilogue(group: int):
        for i in range(group, ntile, 2):
            acc = i % n_acc
            if plant == "group_acc":       # mistake: the two-accumulator indexing kept
                acc = group
            yield (tfull[acc], (i // n_acc) & 1)
            assert acc_tile[acc] == i, "epilogue read another tile's accumulator"
            if fp8:
                s = i % stages
                yield (full[s], (i // stages) & 1)
                assert scale_tile[s] == i, "epilogue read another tile's key scales"
                sfree[s].arrive()
            tempty[acc].arrive()

    roles = [producer()]
    if ntile > 0:   # an item with nothing visible: only thread 0's drain runs
        roles += [mma()] + [epilogue(g) for g in (0, 1) for _ in range(4)]
    ok = run(roles, seed)
    # every copy issued has landed before the CTA exits
    return ok and all(full[s].done == loads[s] for s in range(stages)) and qfull.done == 1


# ---------------------------------------------------------------------------
# attend_tc_kernel: K tiles loaded at once, a tile's buffer refilled with V
# once its score MMAs are done (gather or TMA producers alike), per-tile
# epilogue (two named barriers per tile among the 8 epilogue warps), output
# MMAs after every tile's P rows and V rows, one final commit.  A tile's output
# accumulates in the TMEM columns of its scores (written once every epilogue
# warp has read them: pfull); ranges of five tiles write their P rows into two
# buffers in turn (pempty: the output MMAs of the buffer's previous tile are
# done), shorter ranges into one buffer per tile.

def attend_tc(ntile: int, seed: int, plant: str = "") -> bool:
    q = Bar(1)
    kfull = [Bar(1) for _ in range(ntile)]
    vfull = [Bar(1) for _ in range(ntile)]
    sdone = [Bar(1) for _ in range(ntile)]
    pfull = [Bar(8) for _ in range(ntile)]
    pempty = [Bar(1) for _ in range(2)]
    ofull = Bar(1)
    epi_bar = Bar(8)
    buffer = ["empty"] * ntile
    ring = ntile > 4
    slot = (lambda j: j % 2) if ring else (lambda j: j)
    p_owner = [None] * ntile        # tile whose P rows a buffer holds
    p_read = [True] * ntile         # ... and whether its output MMAs have read them
    s_reads = [0] * ntile           # epilogue warps that have read tile j's score columns

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
            assert s_reads[j] == 8, "output written over scores not yet read"
            assert p_owner[slot(j)] == j, "P rows of another tile"
            p_read[slot(j)] = True
            pempty[j % 2].arrive()
        ofull.arrive()

    def epilogue(me: int):
        for j in range(ntile):
            yield (sdone[j], 0)
            s_reads[j] += 1
            yield from named_barrier(epi_bar, 2 * j)      # the quarters' maxima
            yield from named_barrier(epi_bar, 2 * j + 1)  # the per-head offsets
            if ring and j >= 2 and plant != "pempty":
                yield (pempty[j % 2], (j // 2 - 1) & 1)
            s = slot(j)
            if p_owner[s] != j:
                assert p_read[s], "P rows written over rows still being read"
                p_owner[s], p_read[s] = j, False
            pfull[j].arrive()
        yield from named_barrier(epi_bar, 2 * ntile)      # the sums
        yield from named_barrier(epi_bar, 2 * ntile + 1)  # the coefficients
        yield (ofull, 0)

    return run([producer(), mma()] + [epilogue(w) for w in range(8)], seed)
