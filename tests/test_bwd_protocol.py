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
d = 128, with dS^T packed into S^T's columns. Planted protocol mistakes must
each be caught, so the model is known to be able to fail.
"""
import random

import pytest

# Arrival counts the kernel initialises its barriers with (q_full / q_empty
# are two-slot rings; p_ready and ds_ready take every elementwise thread,
# dq_empty every dQ thread).
CNT = dict(kv_full=1, q_full0=1, q_full1=1, q_empty0=1, q_empty1=1, do_full=1, do_empty=1, s_full=1, dp_full=1,
           p_ready=256, ds_ready=256, dq_full=1, dq_empty=128, acc_done=1)


class Err(Exception):
    """A protocol violation found in one interleaving."""


def run(T, own_dq, new_order, seed, mutation=None, prod_prob=1.0):
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
            st, u = t & 1, t >> 1
            if u >= 1:
                yield ("wait", f"q_empty{st}", u - 1)
            wr(("Q", st), ("Q", t))
            arrive(f"q_full{st}", u, 1)
            yield None
            if t >= 1:
                yield ("wait", "do_empty", t - 1)
            wr("dO", ("dO", t))
            arrive("do_full", t, 1)
            yield None

    def mma(kind, t):
        pipe_q.append(("mma", kind, t))

    def commit(b, k):
        pipe_q.append(("commit", b, k))

    def issuer():
        yield ("wait", "kv_full", 0)
        yield ("wait", "q_full0", 0)
        mma("S", 0); commit("s_full", 0)
        for t in range(T):
            st = t & 1
            if mutation != "dP-skips-dO-wait":
                yield ("wait", "do_full", t)
            if not own_dq and t > 0 and mutation != "dP-skips-dQ-drain":
                yield ("wait", "dq_empty", t - 1)
            mma("dP", t); commit("dp_full", t)
            yield ("wait", "p_ready", t)
            if mutation == "S-before-dV" and t + 1 < T:
                yield ("wait", f"q_full{(t + 1) & 1}", (t + 1) >> 1)
                mma("S", t + 1); commit("s_full", t + 1)
            mma("dV", t); commit("do_empty", t)
            if new_order and mutation != "S-before-dV" and t + 1 < T:
                yield ("wait", f"q_full{(t + 1) & 1}", (t + 1) >> 1)
                mma("S", t + 1); commit("s_full", t + 1)
            yield ("wait", "ds_ready", t)
            mma("dK", t); commit(f"q_empty{st}", t >> 1)
            next_s_first = (not new_order) and own_dq   # main: d = 64 puts S^T(t+1) before dQ
            if next_s_first and t + 1 < T:
                yield ("wait", f"q_full{(t + 1) & 1}", (t + 1) >> 1)
                mma("S", t + 1); commit("s_full", t + 1)
            if own_dq and t > 0:
                yield ("wait", "dq_empty", t - 1)
            mma("dQ", t); commit("dq_full", t)
            if (not new_order) and (not next_s_first) and t + 1 < T:
                yield ("wait", f"q_full{(t + 1) & 1}", (t + 1) >> 1)
                mma("S", t + 1); commit("s_full", t + 1)
            yield None
        commit("acc_done", 0)

    def exec_mma(kind, t):
        if kind == "S":
            rd(("Q", t & 1), ("Q", t)); rd("K", "K")
            for w in W:
                wr(A(w, "lo"), ("S", t)); wr(A(w, "hi"), ("S", t))
        elif kind == "dP":
            rd("dO", ("dO", t))
            for w in W:
                wr(B(w, "lo"), ("dP", t)); wr(B(w, "hi"), ("dP", t))
        elif kind == "dV":
            rd("dO", ("dO", t))
            for w in W:
                rd(A(w, "lo"), ("P", t))
        elif kind == "dK":
            rd(("Q", t & 1), ("Q", t))
            for w in W:
                rd(ds_reg(w), ("dS", t))
        elif kind == "dQ":
            for w in W:
                rd(("smem_dS", w), ("dS", t))
            for w in W:
                wr(DQ(w, "lo"), ("dQ", t)); wr(DQ(w, "hi"), ("dQ", t))

    def ew(w):
        for t in range(T):
            st, u = t & 1, t >> 1
            yield ("wait", f"q_full{st}", u)
            yield ("wait", "s_full", t)
            rd(A(w, "lo"), ("S", t)); wr(A(w, "lo"), ("P_half", t)); yield None
            rd(A(w, "hi"), ("S", t)); wr(A(w, "lo"), ("P", t))
            rd(("Q", st), ("Q", t))  # L slice
            arrive("p_ready", t, 32)
            if mutation != "dS-without-dP-wait":
                yield ("wait", "dp_full", t)
            rd(B(w, "lo"), ("dP", t)); rd(("Q", st), ("Q", t))
            wr(("smem_dS", w), ("dS_half", t)); wr(ds_reg(w), ("dS_half", t))
            yield None
            rd(B(w, "hi"), ("dP", t))
            wr(("smem_dS", w), ("dS", t)); wr(ds_reg(w), ("dS", t))
            arrive("ds_ready", t, 32)
            yield None
        yield ("wait", "acc_done", 0)

    def dqw(q):
        for t in range(T):
            yield ("wait", "dq_full", t)
            for wg in (0, 1):
                w = wg * 4 + q
                rd(DQ(w, "lo"), ("dQ", t)); rd(DQ(w, "hi"), ("dQ", t))
            arrive("dq_empty", t, 32)
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
