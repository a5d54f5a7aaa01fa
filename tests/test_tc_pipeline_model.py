"""Host model of the tensor-core kernel's pipeline protocol (csrc/gemv_tc.cu).

No GPU: the producer, the two MMA chains and the epilogue are generators that
wait on modelled mbarriers (phase parity semantics of mbarrier.try_wait.parity),
and the asynchronous copies and MMAs complete in random order.  The model uses
the kernel's own assignment: stage i of a tile goes to chain i % 2, through a
ring of S/2 slots owned by that chain; the accumulator buffer alternates per
tile and needs both chains' commits.  It checks that no run deadlocks and that
every chain reads the stage it waited for (a waiter two phases ahead of a
slot would see a stale phase as complete and read old data).  The split of a
tile's K stages over a cluster's ranks is checked to partition the stages.
"""
import random

import pytest


class Barrier:
    def __init__(self, count):
        self.count, self.pending, self.phases = count, count, 0

    def arrive(self):
        self.pending -= 1
        if self.pending == 0:
            self.phases += 1
            self.pending = self.count

    def done(self, parity):
        # try_wait.parity(p) succeeds once the phase of parity p has completed
        return (self.phases & 1) != parity


def run_pipeline(stages, stage_counts, seed):
    rng = random.Random(seed)
    sc = stages // 2
    full = [Barrier(1) for _ in range(stages)]
    empty = [Barrier(1) for _ in range(stages)]
    dfull = [Barrier(2) for _ in range(2)]
    dempty = [Barrier(128) for _ in range(2)]
    slot_data, owner = {}, {}

    def producer():
        pos, ph = [0, 0], [0, 0]
        for j, cnt in enumerate(stage_counts):
            for i in range(cnt):
                c = i & 1
                st = c * sc + pos[c]
                while not empty[st].done(ph[c] ^ 1):
                    yield None
                assert owner.setdefault(st, c) == c, "a slot shared by both chains"
                yield ("copy", (st, (j, i)))
                pos[c] += 1
                if pos[c] == sc:
                    pos[c], ph[c] = 0, ph[c] ^ 1

    def chain(c):
        pos, ph = 0, 0
        for j, cnt in enumerate(stage_counts):
            acc = j & 1
            while not dempty[acc].done(((j >> 1) & 1) ^ 1):
                yield None
            for i in range(c, cnt, 2):
                st = c * sc + pos
                while not full[st].done(ph):
                    yield None
                assert slot_data.get(st) == (j, i), "a chain read a stale stage"
                yield ("mma", st)
                pos += 1
                if pos == sc:
                    pos, ph = 0, ph ^ 1
            yield ("commit", acc)

    def epilogue():
        for j, _ in enumerate(stage_counts):
            acc = j & 1
            while not dfull[acc].done((j >> 1) & 1):
                yield None
            for _ in range(128):
                dempty[acc].arrive()
            yield None

    procs = {"producer": producer(), "chain0": chain(0), "chain1": chain(1),
             "epilogue": epilogue()}
    inflight, alive, idle = [], set(procs), 0
    while alive or inflight:
        progressed = False
        if inflight and rng.random() < 0.5:
            kind, payload = inflight.pop(rng.randrange(len(inflight)))
            if kind == "copy":
                st, tag = payload
                slot_data[st] = tag
                full[st].arrive()
            elif kind == "mma":
                empty[payload].arrive()
            else:
                dfull[payload].arrive()
            progressed = True
        if alive:
            name = rng.choice(sorted(alive))
            try:
                step = next(procs[name])
                if step is not None:
                    inflight.append(step)
                    progressed = True
            except StopIteration:
                alive.discard(name)
                progressed = True
        idle = 0 if progressed else idle + 1
        if idle > 20000:
            raise AssertionError(f"deadlock: stages={stages} counts={stage_counts} {alive}")


@pytest.mark.parametrize("stages", [2, 4])
def test_two_chain_pipeline_never_deadlocks_or_reads_stale_stages(stages):
    for seed in range(150):
        rng = random.Random(1000 * stages + seed)
        counts = [rng.choice([0, 1, 1, 2, 3, 4, 5, 7, 8]) for _ in range(rng.randint(1, 9))]
        run_pipeline(stages, counts, seed)


def stage_range(kstages, ks, rank, t):
    """Contiguous K stages of cluster rank `rank` for tile t (the kernel's rule)."""
    per, extra = kstages // ks, kstages % ks
    rr = (rank + t) % ks
    cnt = per + (1 if rr < extra else 0)
    return rr * per + min(rr, extra), cnt


def test_split_k_ranges_partition_the_stages():
    for kstages in range(1, 70):
        for ks in (1, 2, 4, 8):
            if ks > kstages:
                continue
            for t in range(9):
                covered = []
                for rank in range(ks):
                    s0, cnt = stage_range(kstages, ks, rank, t)
                    assert cnt >= 1  # every rank of a cluster has work on every tile
                    covered += range(s0, s0 + cnt)
                assert sorted(covered) == list(range(kstages))
