"""The mbarrier protocols of the tensor-core kernels (indexer_kernel and
attend_tc_kernel) on the CPU: every random interleaving of the warp roles
finishes (no wait that nothing completes) and no buffer is refilled while it
is still read.  The model (tests/_protocol_model.py) restates each role's
waits and arrivals in the kernel's order; planted mistakes show that the
checks bite."""
import random

import pytest

from tests import _protocol_model as M


def test_indexer_protocol_completes_without_hazards():
    """The persistent indexer: random item lists (empty items included),
    stage counts and interleavings, with and without the per-item histogram
    flush."""
    rng = random.Random(0)
    for trial in range(400):
        items = [rng.choice([0, 1, 2, 3, 4, 5, 8, 13, 17]) for _ in range(rng.randint(1, 6))]
        stages = rng.choice([2, 3, 4, 5, 8])
        hist = rng.random() < 0.5
        fp8 = rng.random() < 0.5
        eg = rng.choice([2, 4])
        assert M.indexer(items, stages, trial, hist, fp8=fp8, epi_groups=eg), (items, stages, hist, fp8, eg)


def test_indexer_single_protocol_completes_without_hazards():
    """The one-item decode indexer, bf16 and FP8 keys, two or four TMEM
    accumulators: the first stages are requested before the visibility is
    known, so the visible tile count may fall short of the item's range (down
    to nothing visible)."""
    rng = random.Random(1)
    for trial in range(400):
        cap = rng.choice([0, 1, 2, 3, 4, 5, 8, 13, 17])
        ntile = cap if rng.random() < 0.6 else rng.randint(0, cap)
        stages = rng.choice([2, 3, 5, 8])
        n_acc = rng.choice([2, 4])
        assert M.indexer_single(ntile, stages, trial, fp8=rng.random() < 0.5, cap=cap, n_acc=n_acc), \
            (ntile, cap, stages, n_acc)


def test_indexer_single_wrong_accumulator_is_caught():
    """Four accumulators read with the two-accumulator indexing (buffer =
    epilogue group): the model stalls or reads another tile's accumulator."""
    caught = 0
    for t in range(200):
        try:
            caught += not M.indexer_single(9, 3, t, n_acc=4, plant="group_acc")
        except AssertionError:
            caught += 1
    assert caught == 200


@pytest.mark.parametrize("plant", ["qfree", "wfree", "sfree"])
def test_indexer_missing_item_waits_are_caught(plant):
    """Without the wait for the previous item's MMAs (query rows) or for both
    epilogue groups (head weights), some interleaving refills a buffer that is
    still read, and the model's hazard check fires."""
    # single-tile items: the previous item's end (qfree) does not imply that
    # both groups are done with the item before it
    items = [3, 2, 4, 1, 5] if plant != "wfree" else [2, 1, 1, 1, 2, 1, 1, 1]
    with pytest.raises(AssertionError):
        for t in range(2000):
            M.indexer(items, 3, t, plant=plant, fp8=True)


def test_attend_tc_protocol_completes_without_hazards():
    for ntile in range(1, 6):   # a range with no tile writes its empty result and uses no barrier
        for trial in range(100):
            assert M.attend_tc(ntile, trial), ntile


def test_attend_tc_missing_p_buffer_wait_is_caught():
    # five tiles share two P buffers: without the wait for the output MMAs of
    # a buffer's previous tile, some interleaving overwrites rows still unread
    with pytest.raises(AssertionError):
        for t in range(2000):
            M.attend_tc(5, t, plant="pempty")


def test_planted_mistakes_are_caught(monkeypatch):
    # a buffer-free wait on the wrong parity: the producer waits for a release
    # that only follows its own first load
    def bad_indexer(ntile, stages, seed):
        full = [M.Bar(1) for _ in range(stages)]
        empty = [M.Bar(1) for _ in range(stages)]
        loads = [0] * stages

        def producer():
            for i in range(ntile):
                s, ph = i % stages, (i // stages) & 1
                yield (empty[s], ph)                  # mistake: parity not flipped
                loads[s] += 1
                full[s].arrive()

        def mma():
            for i in range(ntile):
                s, ph = i % stages, (i // stages) & 1
                yield (full[s], ph)
                empty[s].arrive()
        return M.run([producer(), mma()], seed)

    assert not any(bad_indexer(6, 2, t) for t in range(20))   # the producer never starts: caught as a stall

    # the output MMAs not waiting for the V rows: the model's hazard check fires
    def bad_attend(ntile, seed):
        kfull = [M.Bar(1) for _ in range(ntile)]
        sdone = [M.Bar(1) for _ in range(ntile)]
        buffer = ["empty"] * ntile

        def producer():
            for j in range(ntile):
                buffer[j] = "K"
                kfull[j].arrive()
            for j in range(ntile):
                yield (sdone[j], 0)
                buffer[j] = "V"

        def mma():
            for j in range(ntile):
                yield (kfull[j], 0)
                sdone[j].arrive()
            for j in range(ntile):
                assert buffer[j] == "V", "output MMA read K rows"
                yield None
        return M.run([producer(), mma()], seed)

    with pytest.raises(AssertionError):
        for t in range(50):
            bad_attend(3, t)
