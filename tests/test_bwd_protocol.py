"""CPU model check of the backward main kernel's hand-off protocol (no GPU).

`msa_bwd_ws.cuh` runs, per CTA, an info warp, a TMA producer, two MMA issuers,
softmax warps and reduce warps.  They hand off through mbarriers waited by
phase parity:
* an 8-entry task-info ring, released by the reduce warps;
* K/V per bucket segment;
* a two-stage Q/dO ring;
* S/dP in TMEM;
* P/dS in shared memory;
* dQ double-buffered in TMEM;
* dK/dV in TMEM per segment.

This model replays each role's order of waits, arrivals, loads and GEMM
groups under random interleavings (issuer A: S, then dP; issuer B, once its
dQ buffer (and at a segment start dK/dV) is free and then P/dS are stored:
dK, which releases the Q tile, dV, which releases the dO tile, then dQ).  Each issuer's GEMMs complete in its own
issue order, and the two issuers complete in any relative order.  Two softmax
warps stand in for sixteen and two reduce warps for four.  The model asserts
that every parity wait sees the awaited or just-completed phase.  It asserts
that no buffer (info entry, K/V, Q/dO stage, S/dP, P/dS, dQ, dK/dV) is
rewritten before its last reader is done, and that every reader sees the
task's own data.
"""
import random

import pytest

N_SOFT, N_RED, K_INFO = 2, 2, 8


class _Bar:
    def __init__(self, name, count=1):
        self.name, self.done, self.count, self.arr = name, 0, count, 0

    def arrive(self):
        self.arr += 1
        if self.arr == self.count:
            self.arr, self.done = 0, self.done + 1

    def ready_parity(self, parity, k):
        """Wait by parity for the k-th completion (0-based); k = -1 is the
        phase before the first, complete from the start."""
        assert self.done in (k, k + 1), f"parity alias on {self.name}: phase {k}, completed {self.done}"
        assert parity == (k & 1) or k < 0
        return self.done >= k + 1


def _segments(rng, n_tasks):
    seg, out, left = 0, [], 0
    for j in range(n_tasks):
        if left == 0:
            left = rng.randint(1, 5)
            first = True
        else:
            first = False
        left -= 1
        last = left == 0 or j == n_tasks - 1
        out.append((seg, first, last))
        if last:
            seg += 1
            left = 0
    return out


def _simulate(n_tasks, seed, early_do_release=False):
    # early_do_release: a mutation that releases the dO tile with the Q tile
    # after dK, before the dV chain that reads it has run
    rng = random.Random(seed)
    tasks = _segments(rng, n_tasks)
    B = {}
    for n in ["kv", "k_empty", "v_empty", "s_full", "dkv_full"] + [f"q_full{i}" for i in range(2)] + \
             [f"do_full{i}" for i in range(2)] + [f"q_empty{i}" for i in range(2)] + \
             [f"do_empty{i}" for i in range(2)] + ["pds_empty"] + [f"dq_full{i}" for i in range(2)]:
        B[n] = _Bar(n)
    B["s_empty"] = _Bar("s_empty", N_SOFT)
    B["pds_full"] = _Bar("pds_full", N_SOFT)
    for i in range(2):
        B[f"dq_empty{i}"] = _Bar(f"dq_empty{i}", N_RED)
    B["dkv_empty"] = _Bar("dkv_empty", N_RED)
    for i in range(K_INFO):
        B[f"info_full{i}"] = _Bar(f"info_full{i}")
        B[f"info_empty{i}"] = _Bar(f"info_empty{i}", N_RED)

    info = [None] * K_INFO            # task index held by each ring entry
    read_info = {}                    # role -> highest task whose info it has read
    smQ, smDO = [None, None], [None, None]
    smKV = [None]                     # segment held by K/V
    tmSdP = [None]                    # task whose S/dP is in TMEM
    smPdS = [None]
    tmDQ = [None, None]
    tmDKV = [None]                    # segment whose dK/dV accumulate in TMEM
    doneA, doneB = set(), set()       # completed GEMM groups (S/dP; dV/dK and dQ)
    releasedQ, releasedDO = set(), set()  # tasks whose dK / dV completed (Q / dO tile released)
    sdp_read, pds_written = {}, {}    # task -> softmax warps done reading S/dP / writing P/dS
    dq_read, dkv_read = {}, {}        # task / segment -> reduce warps done
    qA, qB, tma = [], [], []

    def note_read(role, j):
        read_info[role] = max(read_info.get(role, -1), j)

    def info_warp():
        for j in range(n_tasks + 1):          # + the sentinel
            slot = j % K_INFO
            k = j // K_INFO - 1                # phase of INFO_EMPTY released by task j-8
            while not B[f"info_empty{slot}"].ready_parity(((j // K_INFO) & 1) ^ 1, k):
                yield
            if j >= K_INFO:
                assert all(read_info.get(r, -1) >= j - K_INFO for r in
                           ["load", "A", "B"] + [f"soft{w}" for w in range(N_SOFT)] +
                           [f"red{w}" for w in range(N_RED)]), "info entry rewritten before every role read it"
            info[slot] = j
            B[f"info_full{slot}"].arrive()
            yield

    def get_info(role, j):
        slot = j % K_INFO
        while not B[f"info_full{slot}"].ready_parity((j // K_INFO) & 1, j // K_INFO):
            yield
        assert info[slot] == j, "info entry overwritten"
        note_read(role, j)

    def producer():
        for j in range(n_tasks):
            yield from get_info("load", j)
            seg, first, last = tasks[j]
            if first:
                while not B["k_empty"].ready_parity((seg & 1) ^ 1, seg - 1):
                    yield
                while not B["v_empty"].ready_parity((seg & 1) ^ 1, seg - 1):
                    yield
                tma.append(("kv", seg))
            st, k = j & 1, (j >> 1) - 1
            while not B[f"q_empty{st}"].ready_parity(((j >> 1) & 1) ^ 1, k):
                yield
            tma.append(("q", j))
            while not B[f"do_empty{st}"].ready_parity(((j >> 1) & 1) ^ 1, k):
                yield
            tma.append(("do", j))
        yield from get_info("load", n_tasks)

    def issuer_a():
        for j in range(n_tasks):
            yield from get_info("A", j)
            seg, first, last = tasks[j]
            st = j & 1
            if first:
                while not B["kv"].ready_parity(seg & 1, seg):
                    yield
            while not B["s_empty"].ready_parity((j & 1) ^ 1, j - 1):
                yield
            while not B[f"q_full{st}"].ready_parity((j >> 1) & 1, j >> 1):
                yield
            qA.append(("S", j))              # S as soon as Q has landed
            while not B[f"do_full{st}"].ready_parity((j >> 1) & 1, j >> 1):
                yield
            qA.append(("dP", j))
        yield from get_info("A", n_tasks)

    def issuer_b():
        for j in range(n_tasks):
            yield from get_info("B", j)
            seg, first, last = tasks[j]
            st = j & 1
            if first:
                while not B["dkv_empty"].ready_parity((seg & 1) ^ 1, seg - 1):
                    yield
            while not B[f"dq_empty{st}"].ready_parity(((j >> 1) & 1) ^ 1, (j >> 1) - 1):
                yield
            while not B["pds_full"].ready_parity(j & 1, j):
                yield
            qB.append(("dK", j))
            qB.append(("dV", j))
            qB.append(("dQ", j))
        yield from get_info("B", n_tasks)

    def softmax(w):
        role = f"soft{w}"
        yield from get_info(role, 0)
        for j in range(n_tasks):
            yield from get_info(role, j + 1)          # look-ahead: the next task's row scalars
            while not B["s_full"].ready_parity(j & 1, j):
                yield
            assert tmSdP[0] == j, "S/dP read before it was computed or after it was overwritten"
            yield
            sdp_read[j] = sdp_read.get(j, 0) + 1
            B["s_empty"].arrive()
            while not B["pds_empty"].ready_parity((j & 1) ^ 1, j - 1):
                yield
            assert j == 0 or (j - 1) in doneB, "P/dS stored over the previous task's before its GEMMs ran"
            smPdS[0] = j
            pds_written[j] = pds_written.get(j, 0) + 1
            B["pds_full"].arrive()
            yield

    def reducer(w):
        role = f"red{w}"
        for j in range(n_tasks):
            yield from get_info(role, j)
            seg, first, last = tasks[j]
            pb = j & 1
            while not B[f"dq_full{pb}"].ready_parity((j >> 1) & 1, j >> 1):
                yield
            assert tmDQ[pb] == j, "dQ read before it was computed or after it was overwritten"
            yield
            dq_read[j] = dq_read.get(j, 0) + 1
            B[f"dq_empty{pb}"].arrive()
            if last:
                while not B["dkv_full"].ready_parity(seg & 1, seg):
                    yield
                assert tmDKV[0] == seg and (j in doneB), "dK/dV read before the segment finished"
                yield
                dkv_read[seg] = dkv_read.get(seg, 0) + 1
                B["dkv_empty"].arrive()
            yield
            B[f"info_empty{j % K_INFO}"].arrive()
        yield from get_info(role, n_tasks)

    def run_a():
        if qA and rng.random() < 0.3:
            kind, j = qA.pop(0)
            seg, first, last = tasks[j]
            assert smKV[0] == seg, "S/dP before its K/V landed"
            assert j == 0 or sdp_read.get(j - 1, 0) == N_SOFT, "S/dP over an S/dP not yet read"
            if kind == "S":
                assert smQ[j & 1] == j, "S before its Q landed"
                return
            assert smQ[j & 1] == j and smDO[j & 1] == j, "dP before its dO landed"
            tmSdP[0] = j
            doneA.add(j)
            B["s_full"].arrive()
            if last:
                B["v_empty"].arrive()

    def run_b():
        if qB and rng.random() < 0.3:
            kind, j = qB.pop(0)
            seg, first, last = tasks[j]
            assert smPdS[0] == j and pds_written.get(j, 0) == N_SOFT, "dV/dK/dQ before P/dS were stored"
            if kind == "dK":
                # dK^T reads the Q tile and dS; the Q tile is released when it completes
                assert smQ[j & 1] == j, "dK after the Q tile was reloaded"
                if first:
                    assert seg == 0 or dkv_read.get(seg - 1, 0) == N_RED, "dK/dV overwritten before drained"
                    tmDKV[0] = seg
                releasedQ.add(j)
                B[f"q_empty{j & 1}"].arrive()
                if early_do_release:
                    B[f"do_empty{j & 1}"].arrive()
                return
            if kind == "dV":
                # dV^T reads the dO tile and P; the dO tile is released when it completes
                assert smDO[j & 1] == j, "dV after the dO tile was reloaded"
                releasedDO.add(j)
                if not early_do_release:
                    B[f"do_empty{j & 1}"].arrive()
                return
            # dQ reads dS and K
            assert smKV[0] == seg, "dQ after K was reloaded"
            assert j < 2 or dq_read.get(j - 2, 0) == N_RED, "dQ over a buffer not yet drained"
            tmDQ[j & 1] = j
            doneB.add(j)
            B["pds_empty"].arrive()
            B[f"dq_full{j & 1}"].arrive()
            if last:
                B["k_empty"].arrive()
                B["dkv_full"].arrive()

    def run_tma():
        if tma and rng.random() < 0.3:
            kind, x = tma.pop(rng.randrange(len(tma)))
            if kind == "kv":
                prev = [t for t in range(n_tasks) if tasks[t][0] == x - 1]
                assert all(t in doneA and t in doneB for t in prev), "K/V reloaded before the segment's GEMMs ran"
                smKV[0] = x
                B["kv"].arrive()
            elif kind == "q":
                assert x < 2 or ((x - 2) in doneA and (x - 2) in releasedQ), "Q stage reloaded too early"
                smQ[x & 1] = x
                B[f"q_full{x & 1}"].arrive()
            else:
                assert x < 2 or ((x - 2) in doneA and (x - 2) in releasedDO), "dO stage reloaded too early"
                smDO[x & 1] = x
                B[f"do_full{x & 1}"].arrive()

    roles = [info_warp(), producer(), issuer_a(), issuer_b()] + [softmax(w) for w in range(N_SOFT)] + \
            [reducer(w) for w in range(N_RED)]
    alive = list(range(len(roles)))
    for _ in range(4 * 10 ** 5):
        if not alive:
            assert not qA and not qB and not tma
            assert len(doneA) == len(doneB) == n_tasks, "a task's GEMMs never ran"
            return
        c = rng.random()
        if c < 0.6:
            i = rng.choice(alive)
            try:
                next(roles[i])
            except StopIteration:
                alive.remove(i)
        else:
            run_a()
            run_b()
            run_tma()
    raise AssertionError("deadlock")


def test_backward_protocol_holds_under_random_schedules():
    rng = random.Random(0)
    for seed in range(400):
        _simulate(rng.randint(1, 24), seed)


def test_protocol_model_catches_an_early_do_release():
    """Releasing the dO tile with the Q tile, after dK, lets the next load
    overwrite dO while the dV chain may still read it, and the model sees it."""
    rng = random.Random(0)
    caught = 0
    for seed in range(200):
        try:
            _simulate(rng.randint(3, 24), seed, early_do_release=True)
        except AssertionError as e:
            assert "reloaded" in str(e)
            caught += 1
    assert caught > 0


def _reduce_staging(flags, seed, dq_commits=True, dq_wait_keep=1):
    """One reduce warp's two staging slots over a task sequence (flags[j]: task
    j ends a bucket segment).  Per task the warp writes both 64-dim dQ halves,
    then a segment end adds four dK/dV chunks; chunk n uses slot n & 1.  A
    chunk read by a bulk reduce-add is committed as its own group (dK/dV
    always; dQ when dq_commits, as the kernel does; a path that read its dQ
    slot back itself would commit none).  Before writing a slot the warp runs
    `cp.async.bulk.wait_group.read N` (N = dq_wait_keep for dQ, 1 for dK/dV):
    afterwards only the N most recently committed groups may still be reading.
    Pending groups finish reading in any order, at random.  Returns the first
    write into a slot that a pending group still reads, or None."""
    rng = random.Random(seed)
    pending = {}  # group index -> slot it reads
    committed = 0
    chunk = 0

    def wait_read(keep):
        for g in [g for g in pending if g < committed - keep]:
            del pending[g]

    def progress():
        for g in list(pending):
            if rng.random() < 0.3:
                del pending[g]

    def use(kind, j, i, keep, commit):
        nonlocal committed, chunk
        progress()
        wait_read(keep)
        if (chunk & 1) in pending.values():
            return (kind, j, i)
        if commit:
            pending[committed] = chunk & 1
            committed += 1
        chunk += 1
        return None

    for j, last in enumerate(flags):
        for hf in range(2):
            bad = use("dq", j, hf, dq_wait_keep, dq_commits)
            if bad:
                return bad
        if last:
            for q in range(4):
                bad = use("dkv", j, q, 1, True)
                if bad:
                    return bad
    return None


def test_reduce_staging_slots_are_never_overwritten_while_read():
    """Every staged chunk is one bulk group and each write waits until at most
    the newest group is still reading, so the slot written (the other one's
    twin) is never still read.  The same wait after a chunk that commits no
    group is not enough (the newest group may be reading the slot about to be
    written), and the model catches that; waiting for every group is."""
    rng = random.Random(1)
    caught = 0
    for seed in range(2000):
        flags = [rng.random() < 0.3 for _ in range(rng.randint(1, 12))]
        assert _reduce_staging(flags, seed) is None
        assert _reduce_staging(flags, seed, dq_commits=False, dq_wait_keep=0) is None
        caught += _reduce_staging(flags, seed, dq_commits=False, dq_wait_keep=1) is not None
    assert caught > 0
