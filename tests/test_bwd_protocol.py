"""Model check of the backward main kernel's synchronisation (fa_bwd.cu,
fa_bwd_main), run on the CPU over random interleavings of its roles.

The roles are the TMA producer, the MMA-issuing thread, the tensor pipe, the
8 elementwise warps and the 4 dQ warps. The tensor pipe executes the issued
MMAs in issue order and fires each commit once every earlier MMA has
executed.

Each role's program is its sequence of mbarrier waits (by phase), arrivals
(with their counts), and reads and writes of TMEM and shared-memory buffers,
as the kernel orders them. Every write stores a (what, tile) version and
every read names the version it needs.

A run fails on any of these:
- a deadlock;
- an arrival for a phase the barrier is not collecting yet;
- a parity wait that finds its barrier two phases ahead (it would block or
  pass wrongly);
- a read that sees another version than it needs.

The issuer waits for all of dS^T before dK (no half-way barrier). Loads can
land late (the producer is held back at random).

Two issue orders are checked. One is the kernel's: S^T(t+1) right after
dV(t), with dS^T packed over the dP^T columns the elementwise warps have
already read. The other is the kernel's earlier order, kept as a second
known-good protocol: S^T(t+1) after dK(t) at d = 64 and after dQ(t) at
d = 128, with dS^T packed into S^T's columns.

At d = dv = 64 the kernel also runs with deeper rings (3 Q slots, 2 dO
slots) and lets other roles vouch for three of the issuing thread's checks:
one elementwise thread checks Q(t+1) before it arrives on p_ready(t) and
dO(t+1) before it arrives on ds_ready(t), and the dQ warps arrive on
ds_ready(t+1) once they have drained dQ(t) (ds_ready then counts 384), so
the thread waits only for p_ready and ds_ready. That protocol is checked
too. Planted protocol mistakes must each be caught, so the model is known
to be able to fail.
"""
import random

import pytest

# Arrival counts the kernel initialises its barriers with (q_full / q_empty
# are two-slot rings; p_ready and ds_ready take every elementwise thread,
# dq_empty every dQ thread).
def counts(nq, ndo, vouch):
    c = dict(kv_full=1, s_full=1, dp_full=1, p_ready=256, ds_ready=256 + (128 if vouch else 0), dq_full=1,
             dq_empty=128, acc_done=1)
    for i in range(nq):
        c[f"q_full{i}"] = c[f"q_empty{i}"] = 1
    for i in range(ndo):
        c[f"do_full{i}"] = c[f"do_empty{i}"] = 1
    return c


class Err(Exception):
    """A protocol violation found in one interleaving."""


def run(T, own_dq, new_order, seed, mutation=None, prod_prob=1.0, vouch=False):
    nq, ndo = (3, 2) if vouch else (2, 1)
    CNT = counts(nq, ndo, vouch)
    rnd = random.Random(seed)
    comp = {b: 0 for b in CNT}
    cur = {b: 0 for b in CNT}
    mem = {}

    def arrive(b, k, n):
        if comp[b] != k:
            raise Err(f"arrival on {b} for phase {k} while collecting {comp[b]}")
        cur[b] += n
        if cur[b] == CNT[b]:
            cur[b] = 0
            comp[b] += 1
        elif cur[b] > CNT[b]:
            raise Err(f"overflow {b}")

    def can_pass(b, k):
        if comp[b] >= k + 2:
            raise Err(f"parity alias on {b}: waiting phase {k}, {comp[b]} done")
        return comp[b] >= k + 1

    def rd(reg, expect):
        got = mem.get(reg)
        if isinstance(expect, set):
            if got not in expect:
                raise Err(f"read {reg}: got {got}, want {expect}")
        elif got != expect:
            raise Err(f"read {reg}: got {got}, want {expect}")

    def wr(reg, val):
        mem[reg] = val

    A = lambda w, h: ("A", w, h)  # TMEM S^T region, warp w's lanes/columns, half h (lo: packed, hi)
    B = lambda w, h: ("B", w, h)  # TMEM dP^T region
    Qd = lambda w, h: ("QD", w, h)  # dQ columns (== B at d = 128)
    DQ = (lambda w, h: B(w, h)) if not own_dq else Qd
    ds_reg = (lambda w: B(w, "lo")) if new_order else (lambda w: A(w, "hi"))
    if mutation == "dS-left-in-S-region":
        ds_reg = lambda w: A(w, "hi")
    W = range(8)

    # Programs: generators that yield ("wait", barrier, phase) to block, or
    # None to let another role run.
    pipe_q = []  # issued MMAs / commits, executed in order

    def producer():
        wr("K", "K")
        arrive("kv_full", 0, 1)
        for t in range(T):
            st, u = t % nq, t // nq
            if u >= 1:
                yield ("wait", f"q_empty{st}", u - 1)
            wr(("Q", st), ("Q", t))
            arrive(f"q_full{st}", u, 1)
            yield None
            so, uo = t % ndo, t // ndo
            if uo >= 1:
                yield ("wait", f"do_empty{so}", uo - 1)
            wr(("dO", so), ("dO", t))
            arrive(f"do_full{so}", uo, 1)
            yield None

    def mma(kind, t):
        pipe_q.append(("mma", kind, t))

    def commit(b, k):
        pipe_q.append(("commit", b, k))

    def wait_q(t):  # the issuer's own check of Q(t) (none where it is vouched for)
        if not vouch:
            yield ("wait", f"q_full{t % nq}", t // nq)

    def issuer():
        yield ("wait", "kv_full", 0)
        yield ("wait", "q_full0", 0)
        mma("S", 0); commit("s_full", 0)
        for t in range(T):
            st = t % nq
            if mutation != "dP-skips-dO-wait" and (not vouch or t == 0):
                yield ("wait", f"do_full{t % ndo}", t // ndo)
            if not own_dq and t > 0 and mutation != "dP-skips-dQ-drain":
                yield ("wait", "dq_empty", t - 1)
            mma("dP", t); commit("dp_full", t)
            yield ("wait", "p_ready", t)
            if mutation == "S-before-dV" and t + 1 < T:
                yield from wait_q(t + 1)
                mma("S", t + 1); commit("s_full", t + 1)
            mma("dV", t); commit(f"do_empty{t % ndo}", t // ndo)
            if new_order and mutation != "S-before-dV" and t + 1 < T:
                yield from wait_q(t + 1)
                mma("S", t + 1); commit("s_full", t + 1)
            yield ("wait", "ds_ready", t)
            mma("dK", t); commit(f"q_empty{st}", t // nq)
            next_s_first = (not new_order) and own_dq   # main: d = 64 puts S^T(t+1) before dQ
            if next_s_first and t + 1 < T:
                yield from wait_q(t + 1)
                mma("S", t + 1); commit("s_full", t + 1)
            if own_dq and t > 0 and not vouch:
                yield ("wait", "dq_empty", t - 1)
            mma("dQ", t); commit("dq_full", t)
            if (not new_order) and (not next_s_first) and t + 1 < T:
                yield from wait_q(t + 1)
                mma("S", t + 1); commit("s_full", t + 1)
            yield None
        commit("acc_done", 0)

    def exec_mma(kind, t):
        if kind == "S":
            rd(("Q", t % nq), ("Q", t)); rd("K", "K")
            for w in W:
                wr(A(w, "lo"), ("S", t)); wr(A(w, "hi"), ("S", t))
        elif kind == "dP":
            rd(("dO", t % ndo), ("dO", t))
            for w in W:
                wr(B(w, "lo"), ("dP", t)); wr(B(w, "hi"), ("dP", t))
        elif kind == "dV":
            rd(("dO", t % ndo), ("dO", t))
            for w in W:
                rd(A(w, "lo"), ("P", t))
        elif kind == "dK":
            rd(("Q", t % nq), ("Q", t))
            for w in W:
                rd(ds_reg(w), ("dS", t))
        elif kind == "dQ":
            for w in W:
                rd(("smem_dS", w), ("dS", t))
            for w in W:
                wr(DQ(w, "lo"), ("dQ", t)); wr(DQ(w, "hi"), ("dQ", t))

    def ew(w):
        for t in range(T):
            st, u = t % nq, t // nq
            yield ("wait", f"q_full{st}", u)
            yield ("wait", "s_full", t)
            rd(A(w, "lo"), ("S", t)); wr(A(w, "lo"), ("P_half", t)); yield None
            rd(A(w, "hi"), ("S", t)); wr(A(w, "lo"), ("P", t))
            rd(("Q", st), ("Q", t))  # L slice
            if vouch and w == 0 and t + 1 < T and mutation != "vouch-skips-Q-check":
                yield ("wait", f"q_full{(t + 1) % nq}", (t + 1) // nq)  # vouches for S^T(t+1)
            arrive("p_ready", t, 32)
            if mutation != "dS-without-dP-wait":
                yield ("wait", "dp_full", t)
            rd(B(w, "lo"), ("dP", t)); rd(("Q", st), ("Q", t))
            wr(("smem_dS", w), ("dS_half", t)); wr(ds_reg(w), ("dS_half", t))
            yield None
            rd(B(w, "hi"), ("dP", t))
            wr(("smem_dS", w), ("dS", t)); wr(ds_reg(w), ("dS", t))
            if vouch and w == 0 and t + 1 < T and mutation != "vouch-skips-dO-check":
                yield ("wait", f"do_full{(t + 1) % ndo}", (t + 1) // ndo)  # vouches for dP^T(t+1)
            arrive("ds_ready", t, 32)
            yield None
        yield ("wait", "acc_done", 0)

    def dqw(q):
        if vouch:
            arrive("ds_ready", 0, 32)  # nothing to drain before dQ(0)
        for t in range(T):
            yield ("wait", "dq_full", t)
            if vouch and mutation == "vouch-dQ-arrives-before-drain" and t + 1 < T:
                arrive("ds_ready", t + 1, 32)
                yield None
            for wg in (0, 1):
                w = wg * 4 + q
                rd(DQ(w, "lo"), ("dQ", t)); rd(DQ(w, "hi"), ("dQ", t))
            if not vouch:
                arrive("dq_empty", t, 32)
            elif t + 1 < T and mutation != "vouch-dQ-arrives-before-drain":
                arrive("ds_ready", t + 1, 32)  # vouches for dQ(t+1)'s columns
            yield None

    procs = {"prod": producer(), "mma": issuer()}
    for w in W:
        procs[f"ew{w}"] = ew(w)
    for q in range(4):
        procs[f"dq{q}"] = dqw(q)
    pending = {n: None for n in procs}  # the wait a process is blocked on
    done = set()
    steps = 0
    while True:
        steps += 1
        if steps > 200000:
            raise Err("livelock")
        ready = []
        for n, g in procs.items():
            if n in done:
                continue
            pw = pending[n]
            if pw is None or can_pass(pw[1], pw[2]):
                ready.append(n)
        if pipe_q:
            ready.append("pipe")
        if "prod" in ready and len(ready) > 1 and rnd.random() >= prod_prob:
            ready.remove("prod")  # prod_prob < 1 makes loads land late
        if not ready:
            if len(done) == len(procs):
                return
            raise Err("deadlock: " + ", ".join(f"{n}@{pending[n]}" for n in procs if n not in done))
        n = rnd.choice(ready)
        if n == "pipe":
            op = pipe_q.pop(0)
            if op[0] == "mma":
                exec_mma(op[1], op[2])
            else:
                arrive(op[1], op[2], 1)
            continue
        pending[n] = None
        try:
            ev = next(procs[n])
            if ev is not None:
                pending[n] = ev
        except StopIteration:
            done.add(n)



ORDERS = {"kernel": True, "earlier": False}


@pytest.mark.parametrize("order", sorted(ORDERS))
@pytest.mark.parametrize("d", [64, 128])
def test_protocol_is_free_of_deadlock_aliasing_and_hazards(order, d):
    for T in (1, 2, 3, 4, 5, 7):
        for seed in range(60):
            run(T, own_dq=(d == 64), new_order=ORDERS[order], seed=seed, prod_prob=0.15 if seed % 3 == 0 else 1.0)


def test_vouched_protocol_at_d64_is_free_of_deadlock_aliasing_and_hazards():
    for T in (1, 2, 3, 4, 5, 6, 7, 9):
        for seed in range(80):
            run(T, own_dq=True, new_order=True, seed=seed, prod_prob=(0.1, 0.4, 1.0)[seed % 3], vouch=True)


@pytest.mark.parametrize("mutation", [
    "vouch-skips-Q-check",            # S^T(t+1) would read a Q tile that has not landed
    "vouch-skips-dO-check",           # dP^T(t+1) would read a dO tile that has not landed
    "vouch-dQ-arrives-before-drain",  # dQ(t+1) would overwrite dQ(t) before its drain
    "dP-skips-dO-wait",               # dP^T(0) would read a dO tile that has not landed
])
def test_planted_mistakes_in_the_vouched_protocol_are_caught(mutation):
    failures = 0
    for T in (2, 3, 4, 5):
        for seed in range(60):
            try:
                run(T, own_dq=True, new_order=True, seed=seed, mutation=mutation, prod_prob=0.1 if seed & 1 else 0.5,
                    vouch=True)
            except Err:
                failures += 1
    assert failures > 0, f"{mutation} went unnoticed"


@pytest.mark.parametrize("mutation, order, d", [
    ("dS-left-in-S-region", "kernel", 128),       # S^T(t+1) would overwrite dS^T(t) before dK(t)
    ("S-before-dV", "kernel", 128),               # S^T(t+1) would overwrite P^T(t) before dV(t)
    ("dP-skips-dQ-drain", "kernel", 128),         # dP^T(t+1) would overwrite dQ(t) before its drain
    ("dP-skips-dQ-drain", "earlier", 128),
    ("dS-without-dP-wait", "kernel", 64),         # dS phase would read dP^T before it is written
    ("dP-skips-dO-wait", "kernel", 128),          # dP^T(t) would read a dO tile that has not landed
])
def test_planted_protocol_mistakes_are_caught(mutation, order, d):
    failures = 0
    for T in (2, 3, 4):
        for seed in range(40):
            try:
                run(T, own_dq=(d == 64), new_order=ORDERS[order], seed=seed, mutation=mutation,
                    prod_prob=0.15 if seed & 1 else 1.0)
            except Err:
                failures += 1
    assert failures > 0, f"{mutation} went unnoticed"
