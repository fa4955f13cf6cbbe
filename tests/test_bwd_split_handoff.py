"""Model check of the hand-off between the two halves of a split backward
work item (fa_bwd.cu, fa_bwd_main's dV / dK epilogue), run on the CPU over
random interleavings.

Without a causal mask a short last round of key tiles runs each tile as two
CTAs, each over half of the tile's query tiles. Each half's epilogue threads:
  1. write their fp32 dV / dK rows to the half's partial area (plain stores),
  2. fence (`__threadfence`), then meet on a named barrier,
  3. one thread takes a ticket (`atomicAdd` on the item's counter, zeroed by
     the preprocess kernel of the same call), and a second named barrier
     hands the ticket to every thread,
  4. the half that drew ticket 1 fences again, reads the other half's rows,
     adds them to its own and stores the item's dV and dK; the other half
     stops. Neither half ever waits for the other.

Memory model: a thread's stores sit in its own buffer and drain to global
memory one at a time at random moments, in any order; a fence drains them
all. The atomic and the reads see global memory. The partial area starts
with the previous call's values, so a read that comes too early sees stale
rows. A run fails if the finishing half reads a stale or missing partner
row, if no half or both halves finish, or if the stored item is not the sum
of both halves. Planted mistakes must each be caught.
"""
import random

import pytest

ROWS = 4  # epilogue threads per half (one partial row each)


class Err(Exception):
    pass


def run(seed, calls=2, mutation=None):
    rnd = random.Random(seed)
    mem = {}  # global memory: ("part", half, row) -> (call, value); ("cnt",) -> int; ("out", row) -> value
    for r in range(ROWS):
        for h in range(2):
            mem[("part", h, r)] = (-1, 0.0)  # left over from an earlier call
    mem[("cnt",)] = 0
    for call in range(calls):
        if mutation != "counter-not-zeroed":
            mem[("cnt",)] = 0  # the preprocess kernel of this call
        for r in range(ROWS):
            mem.pop(("out", r), None)
        own = {(h, r): float(10 * call + 2 * r + h + 1) for h in range(2) for r in range(ROWS)}
        buf = {(h, r): [] for h in range(2) for r in range(ROWS)}  # pending stores per thread
        ticket = {}
        # per-thread programs as generators of steps; barriers are modelled by
        # counters that a step waits on (a blocked step is retried later)
        arrived = {(h, b): 0 for h in range(2) for b in (1, 2)}

        def drain_one(key):
            if buf[key]:
                i = rnd.randrange(len(buf[key]))
                addr, val = buf[key].pop(i)
                mem[addr] = val

        def fence(key):
            while buf[key]:
                drain_one(key)

        def thread(h, r):
            key = (h, r)
            buf[key].append((("part", h, r), (call, own[key])))
            yield
            if mutation != "no-writer-fence":
                fence(key)
            if mutation == "ticket-before-barrier" and r == 0:
                ticket[h] = mem[("cnt",)]
                mem[("cnt",)] += 1
                yield
            arrived[(h, 1)] += 1
            while arrived[(h, 1)] < ROWS:
                yield
            if mutation != "ticket-before-barrier" and r == 0:
                ticket[h] = mem[("cnt",)]  # atomicAdd returns the old value
                mem[("cnt",)] += 1
            arrived[(h, 2)] += 1
            while arrived[(h, 2)] < ROWS:
                yield
            finish = ticket[h] == (0 if mutation == "first-finishes" else 1)
            if not finish:
                return
            fence(key)
            yield
            got = mem[("part", 1 - h, r)]
            if got[0] != call:
                raise Err(f"call {call}: half {h} row {r} read a stale partner row {got}")
            buf[key].append((("out", r), own[key] + got[1]))
            fence(key)

        live = [thread(h, r) for h in range(2) for r in range(ROWS)]
        keys = [(h, r) for h in range(2) for r in range(ROWS)]
        for g in live:
            next(g)
        steps = 0
        while live:
            steps += 1
            if steps > 10000:
                raise Err("no progress")
            if rnd.random() < 0.3:  # some store drains on its own
                drain_one(rnd.choice(keys))
            i = rnd.randrange(len(live))
            try:
                next(live[i])
            except StopIteration:
                live.pop(i)
        for key in keys:
            fence(key)
        finishers = [h for h in range(2) if ticket.get(h) == (0 if mutation == "first-finishes" else 1)]
        if len(finishers) != 1:
            raise Err(f"call {call}: {len(finishers)} halves finished the item (tickets {ticket})")
        for r in range(ROWS):
            want = own[(0, r)] + own[(1, r)]
            if mem.get(("out", r)) != want:
                raise Err(f"call {call}: row {r} stored {mem.get(('out', r))}, want {want}")


def test_handoff_sums_both_halves_in_every_interleaving():
    for seed in range(2000):
        run(seed)


@pytest.mark.parametrize("mutation", ["no-writer-fence", "ticket-before-barrier", "first-finishes",
                                      "counter-not-zeroed"])
def test_planted_handoff_mistakes_are_caught(mutation):
    caught = 0
    for seed in range(2000):
        try:
            run(seed, mutation=mutation)
        except Err:
            caught += 1
    assert caught > 0, f"mutation {mutation} was never caught"
