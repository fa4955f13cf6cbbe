"""Model check of the forward kernel's synchronisation (fa_fwd.cu,
fa_fwd_kernel), run on the CPU over random interleavings of its roles.

The kernel is persistent: one CTA walks a sequence of work items, each two
query tiles A and B with key-tile ranges [kb, ke), and every barrier phase
and K/V ring position runs on from one item to the next. The model's roles
are the TMA producer, the copy engine (each issued load lands at a random
later moment), the MMA-issuing thread, the tensor pipe (executes the issued
MMAs in order; a commit arrives once every earlier MMA has executed) and the
8 softmax warps (4 per tile, 32 arrivals each).

Every buffer write stores a version and every read names the version it
needs: Q_X = (item), K/V slot = (item, key tile), S/P_X per warp = (item,
key tile), O_X per warp = (item, last key tile accumulated). A run fails on a
deadlock, an arrival for a phase the barrier is not collecting, a parity wait
that finds its barrier two phases ahead, or a read of the wrong version.

The issuing thread checks K_j / V_j only where nothing else vouches for
them: tile B's S uses the key tile tile A has just waited for, and with a
4-deep K/V ring (NS >= 3, as in the kernel) the softmax of tile X checks the
next key tile's K / V before it arrives on P_X's barrier, so inside an item
the issuer's wait for P_X(j-1) also covers S_X(j).

Item sequences are random but keep the kernel's invariants: tile B's range
starts and ends no earlier than A's and starts no later than A's end; either
range may be empty. Planted protocol mistakes must each be caught, so the
model is known to be able to fail.
"""
import random

import pytest


class Err(Exception):
    """A protocol violation found in one interleaving."""


def random_items(rnd, n_items):
    items = []
    for _ in range(n_items):
        kind = rnd.randrange(6)
        if kind == 0:  # both empty (rows that see no key)
            items.append(((0, 0), (0, 0)))
            continue
        a0 = rnd.randrange(0, 3)
        a1 = a0 + rnd.randrange(1, 4)
        if kind == 1:  # A empty, B not
            b0 = rnd.randrange(0, 3)
            items.append(((0, 0), (b0, b0 + rnd.randrange(1, 4))))
        elif kind == 2:  # no tile B (past the last row) or B empty
            items.append(((a0, a1), (0, 0)))
        else:
            b0 = rnd.randrange(a0, a1 + 1)
            b1 = max(a1, b0 + 1) + rnd.randrange(0, 2)
            items.append(((a0, a1), (b0, b1)))
    return items


def run(items, NS, seed, mutation=None, copy_prob=1.0):
    rnd = random.Random(seed)
    kv_soft = NS >= 3
    cnt = {"drain": 1}
    for x in (0, 1):
        cnt.update({f"q_full{x}": 1, f"q_empty{x}": 1, f"s_full{x}": 1, f"p_full{x}": 128, f"o_done{x}": 1})
    for s in range(NS):
        cnt.update({f"kv_full{s}": 1, f"k_empty{s}": 1, f"v_empty{s}": 1})
    comp = {b: 0 for b in cnt}
    cur = {b: 0 for b in cnt}
    tx = {b: 0 for b in cnt}
    mem = {}

    def maybe_complete(b):
        if cur[b] == cnt[b] and tx[b] == 0:
            cur[b] = 0
            comp[b] += 1

    def arrive(b, k, n, add_tx=0):
        if comp[b] != k:
            raise Err(f"arrival on {b} for phase {k} while collecting {comp[b]}")
        cur[b] += n
        tx[b] += add_tx
        if cur[b] > cnt[b]:
            raise Err(f"overflow {b}")
        maybe_complete(b)

    def can_pass(b, k):
        if comp[b] >= k + 2:
            raise Err(f"parity alias on {b}: waiting phase {k}, {comp[b]} done")
        return comp[b] >= k + 1

    def rd(reg, expect):
        if mem.get(reg) != expect:
            raise Err(f"read {reg}: got {mem.get(reg)}, want {expect}")

    def wr(reg, val):
        mem[reg] = val

    active = lambda it, x, j: it[x][0] <= j < it[x][1]
    union = lambda it: ((it[0][0] if it[0][1] > it[0][0] else it[1][0]), max(it[0][1], it[1][1]))
    W = range(4)

    copies = []  # loads in flight: (buffer, version, barrier)

    def load(buf, ver, bar):
        copies.append((buf, ver, bar))

    def producer():
        nq = [0, 0]
        g = 0
        for n, it in enumerate(items):
            ub, ue = union(it)
            for x in (0, 1):
                if it[x][1] <= it[x][0]:
                    continue
                if nq[x] > 0 and mutation != "q-load-skips-q_empty":
                    yield ("wait", f"q_empty{x}", nq[x] - 1)
                arrive(f"q_full{x}", nq[x], 1, add_tx=1)
                load(("Q", x), n, (f"q_full{x}", nq[x]))
                nq[x] += 1
                yield None
            for jj in range(ue - ub):
                s, u = g % NS, g // NS
                if u >= 1:
                    yield ("wait", f"k_empty{s}", u - 1)
                arrive(f"kv_full{s}", u, 1, add_tx=2)
                load(("K", s), (n, ub + jj), (f"kv_full{s}", u))
                yield None
                if u >= 1:
                    yield ("wait", f"v_empty{s}", u - 1)
                load(("V", s), (n, ub + jj), (f"kv_full{s}", u))
                g += 1
                yield None

    pipe_q = []

    def issuer():
        nq = [0, 0]
        np_ = [0, 0]
        base = 0
        for n, it in enumerate(items):
            ub, ue = union(it)

            def issue_s(x, j, wait_kv):
                pos = base + j - ub
                s = pos % NS
                if j == it[x][0]:
                    yield ("wait", f"q_full{x}", nq[x])
                    nq[x] += 1
                if wait_kv:
                    yield ("wait", f"kv_full{s}", pos // NS)
                pipe_q.append(("S", n, x, j, s))
                pipe_q.append(("commit", f"s_full{x}"))
                last = it[x][0] if mutation == "q_empty-after-first-S" else it[x][1] - 1
                if j == last:
                    pipe_q.append(("commit", f"q_empty{x}"))

            def issue_pv(x, j):
                s = (base + j - ub) % NS
                yield ("wait", f"p_full{x}", np_[x])
                np_[x] += 1
                pipe_q.append(("PV", n, x, j, s))

            if ue > ub:
                for x in (0, 1):
                    if active(it, x, ub):
                        yield from issue_s(x, ub, not (x == 1 and active(it, 0, ub)))
                pipe_q.append(("commit", f"k_empty{base % NS}"))
            for j in range(ub, ue):
                for x in (0, 1):
                    last_pv = active(it, x, j) and not active(it, x, j + 1)
                    if last_pv and mutation == "o_done-before-last-PV":
                        pipe_q.append(("commit", f"o_done{x}"))
                    if active(it, x, j):
                        yield from issue_pv(x, j)
                        if x == 1 or not active(it, 1, j):
                            pipe_q.append(("commit", f"v_empty{(base + j - ub) % NS}"))
                    if active(it, x, j + 1):
                        covered = ((x == 1 and active(it, 0, j + 1) and (not kv_soft or active(it, 0, j)))
                                   or (kv_soft and active(it, x, j)))
                        if mutation == "issuer-trusts-uncovered-kv":
                            covered = True
                        yield from issue_s(x, j + 1, not covered)
                        if x == 1 or not active(it, 1, j + 1):
                            pipe_q.append(("commit", f"k_empty{(base + j + 1 - ub) % NS}"))
                    elif last_pv and mutation != "o_done-before-last-PV":
                        pipe_q.append(("commit", f"o_done{x}"))
                yield None
            base += ue - ub
        pipe_q.append(("commit", "drain"))

    def exec_op(op):
        kind = op[0]
        if kind == "S":
            _, n, x, j, s = op
            rd(("Q", x), n)
            rd(("K", s), (n, j))
            for w in W:
                wr(("S", x, w), (n, j))
        elif kind == "PV":
            _, n, x, j, s = op
            rd(("V", s), (n, j))
            for w in W:
                rd(("P", x, w), (n, j))
                if j > items[n][x][0]:
                    rd(("O", x, w), (n, j - 1))
                wr(("O", x, w), (n, j))

    def softmax(x, w):
        ns = no = 0
        base = 0
        deferred = None  # mutation "epilogue-after-next-P": the O read put off past the next P
        for n, it in enumerate(items):
            ub, ue = union(it)
            item_base = base
            base += ue - ub
            kb, ke = it[x]
            for j in range(kb, ke):
                yield ("wait", f"s_full{x}", ns)
                ns += 1
                rd(("S", x, w), (n, j))
                wr(("P", x, w), (n, j))
                yield None
                if j > kb:  # a lazy rescale of the O row (taken or not, it must be safe)
                    rd(("O", x, w), (n, j - 1))
                if kv_soft and w == 0 and j + 1 < ke and mutation != "softmax-skips-kv-check":
                    pos = item_base + j + 1 - ub
                    yield ("wait", f"kv_full{pos % NS}", pos // NS)
                arrive(f"p_full{x}", ns - 1, 32)
                yield None
                if deferred is not None:
                    rd(*deferred)
                    deferred = None
            if ke > kb:
                if mutation != "epilogue-skips-o_done":
                    yield ("wait", f"o_done{x}", no)
                no += 1
                if mutation == "epilogue-after-next-P":
                    deferred = (("O", x, w), (n, ke - 1))
                else:
                    rd(("O", x, w), (n, ke - 1))
                yield None
        if deferred is not None:
            rd(*deferred)

    procs = {"prod": producer(), "mma": issuer()}
    for x in (0, 1):
        for w in W:
            procs[f"sm{x}{w}"] = softmax(x, w)
    pending = {n: None for n in procs}
    done = set()
    steps = 0
    while True:
        steps += 1
        if steps > 400000:
            raise Err("livelock")
        ready = [n for n in procs if n not in done and (pending[n] is None or can_pass(pending[n][1], pending[n][2]))]
        if pipe_q:
            ready.append("pipe")
        if copies and (not ready or rnd.random() < copy_prob):
            ready.append("copy")  # copy_prob < 1 makes loads land late
        if not ready:
            if len(done) == len(procs):
                if comp["drain"] != 1:
                    raise Err("drain never fired")
                return
            raise Err("deadlock: " + ", ".join(f"{n}@{pending[n]}" for n in procs if n not in done))
        n = rnd.choice(ready)
        if n == "pipe":
            op = pipe_q.pop(0)
            if op[0] == "commit":
                b = op[1]
                arrive(b, comp[b], 1)
            else:
                exec_op(op)
            continue
        if n == "copy":
            buf, ver, (bar, k) = copies.pop(rnd.randrange(len(copies)))
            wr(buf, ver)
            if comp[bar] != k:
                raise Err(f"copy completes {bar} phase {k} while collecting {comp[bar]}")
            tx[bar] -= 1
            maybe_complete(bar)
            continue
        pending[n] = None
        try:
            ev = next(procs[n])
            if ev is not None:
                pending[n] = ev
        except StopIteration:
            done.add(n)


@pytest.mark.parametrize("NS", [2, 4])
def test_protocol_is_free_of_deadlock_aliasing_and_hazards(NS):
    rnd = random.Random(NS)
    for trial in range(120):
        items = random_items(rnd, rnd.randrange(1, 6))
        for seed in range(6):
            run(items, NS, seed=trial * 100 + seed, copy_prob=0.1 if seed % 3 == 0 else 1.0)


def test_causal_pairs_and_full_rows():
    # the two shapes the headline workloads produce: causal pairs (A one key tile
    # shorter than B) and full rows (A and B over the same range)
    causal = [((0, 2 * m + 1), (0, 2 * m + 2)) for m in (3, 0, 2, 1)]
    full = [((0, 3), (0, 3))] * 3
    for NS in (2, 4):
        for items in (causal, full, causal + full):
            for seed in range(40):
                run(items, NS, seed)


@pytest.mark.parametrize("mutation, NS", [
    ("q-load-skips-q_empty", 2),        # the next item's Q would land while S of this item still reads it
    ("q_empty-after-first-S", 2),       # Q released after its first S instead of its last
    ("epilogue-skips-o_done", 2),       # the epilogue would read O before the last P.V
    ("o_done-before-last-PV", 2),       # o_done committed before the last P.V is issued
    ("epilogue-after-next-P", 4),       # the next item's first P.V would overwrite O before the epilogue reads it
    ("softmax-skips-kv-check", 4),      # S(j+1) would read a K tile that has not landed
    ("issuer-trusts-uncovered-kv", 4),  # tile B's first S inside an item, with no P barrier vouching for its K
])
def test_planted_protocol_mistakes_are_caught(mutation, NS):
    rnd = random.Random(7)
    failures = 0
    # random item sequences, plus one where tile B starts exactly where tile A ends
    lists = [random_items(rnd, rnd.randrange(2, 5)) for _ in range(60)] + [[((0, 2), (2, 4)), ((0, 1), (1, 3))] * 2] * 40
    for trial, items in enumerate(lists):
        for seed in range(4):
            try:
                run(items, NS, seed=trial * 10 + seed, mutation=mutation, copy_prob=0.2 if seed & 1 else 1.0)
            except Err:
                failures += 1
    assert failures > 0, f"{mutation} went unnoticed"
