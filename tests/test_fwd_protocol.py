"""CPU model check of the forward kernel's hand-off protocol (no GPU).

The forward (`msa_fwd.cu`) runs one load/MMA warp and four softmax warps per
CTA that hand off through mbarriers waited by phase parity.  A parity wait is
correct only while the barrier is on the awaited phase or has just completed
it; one phase behind passes too early, two phases ahead never passes.  This
model replays the kernel's order of waits, arrivals, GEMM issues and TMA loads
under random interleavings.  The MMA pipe completes in issue order and TMA
loads land in any order.  It asserts that every wait sees an allowed phase
and that no buffer is overwritten before its reader has finished.  Two
variants of the protocol fail it.  In one, the softmax warps wait only for the
last P V of an item.  The other also has a single P-written barrier for both
S/P buffers.
"""
import random

import pytest


class _Bar:
    def __init__(self, name, count=1):
        self.name, self.done, self.count, self.arr = name, 0, count, 0

    def arrive(self):
        self.arr += 1
        if self.arr == self.count:
            self.arr, self.done = 0, self.done + 1

    def ready(self, k):
        """Wait for the k-th completion (0-based) by parity, as the kernel does."""
        assert self.done in (k, k + 1), f"parity alias on {self.name}: phase {k}, completed {self.done}"
        return self.done == k + 1


def _simulate(items, seed, n_softmax=2, split_pfull=True, in_order_pv=True):
    """One S buffer, two P buffers and O in TMEM; K and V double-buffered."""
    rng = random.Random(seed)
    B = {n: _Bar(n) for n in ["q", "pv", "s", "k0", "k1", "v0", "v1"]}
    B["sfree"] = _Bar("sfree", n_softmax)
    pf = ["pf0", "pf1"] if split_pfull else ["pf", "pf"]
    for n in set(pf):
        B[n] = _Bar(n, n_softmax)
    mma_q, tma = [], []
    smK, smV, tmP = {0: None, 1: None}, {0: None, 1: None}, {0: None, 1: None}
    tmS = [None]
    done_S, done_PV = set(), set()

    def pf_phase(n):
        return n >> 1 if split_pfull else n

    def issuer():
        seq, ph_q = 0, 0
        for nblk in items:
            seq0 = seq
            yield "sync"
            if nblk > 0:
                tma.append(("q", None, "Q", None))
                for j in range(min(2, nblk)):
                    n = seq0 + j
                    tma.append((f"k{n & 1}", n & 1, "K", n))
                    tma.append((f"v{n & 1}", n & 1, "V", n))
                while not B["q"].ready(ph_q):
                    yield None
                ph_q += 1
                while not B[f"k{seq0 & 1}"].ready(seq0 >> 1):
                    yield None
                mma_q.append(("S", seq0))
                for j in range(nblk):
                    n, bf = seq0 + j, (seq0 + j) & 1
                    if j + 1 < nblk:          # S_{j+1}: K landed, every warp has read S_j
                        while not B[f"k{(n + 1) & 1}"].ready((n + 1) >> 1):
                            yield None
                        while not B["sfree"].ready(n):
                            yield None
                        mma_q.append(("S", n + 1))
                        if j + 2 < nblk:      # K_{j+2} where K_j was (S_j done)
                            tma.append((f"k{bf}", bf, "K", n + 2))
                    if j >= 1 and j + 1 < nblk:   # V_{j+1} once P V of block j-1 is done
                        while not B["pv"].ready(n - 1):
                            yield None
                        tma.append((f"v{bf ^ 1}", bf ^ 1, "V", n + 1))
                    while not B[pf[bf]].ready(pf_phase(n)):
                        yield None
                    while not B[f"v{bf}"].ready(n >> 1):
                        yield None
                    mma_q.append(("PV", n))
            seq = seq0 + nblk
            yield "sync"

    def softmax():
        seq = 0
        for nblk in items:
            seq0 = seq
            yield "sync"
            for j in range(nblk):
                n, bf = seq0 + j, (seq0 + j) & 1
                while not B["s"].ready(n):
                    yield None
                assert tmS[0] == n, "S_j overwritten before it was read"
                yield None
                B["sfree"].arrive()
                yield None
                if j > 0 and rng.random() < 0.3:      # O rescale
                    while not B["pv"].ready(n - 1):
                        yield None
                    assert (n - 1) in done_PV and n not in done_PV
                assert n < 2 or (n - 2) in done_PV, "P stored over a P not yet read"
                tmP[bf] = n
                if j > 0 and in_order_pv:
                    while not B["pv"].ready(n - 1):
                        yield None
                B[pf[bf]].arrive()
                yield None
            if nblk > 0:
                while not B["pv"].ready(seq0 + nblk - 1):
                    yield None
                assert (seq0 + nblk - 1) in done_PV      # epilogue reads the finished O
            seq = seq0 + nblk
            yield "sync"

    def mma_step():
        if mma_q and rng.random() < 0.3:
            kind, n = mma_q.pop(0)
            if kind == "S":
                assert smK[n & 1] == n, "S before its K landed"
                assert B["sfree"].done >= n, "S over an S not yet read"
                tmS[0] = n
                done_S.add(n)
                B["s"].arrive()
            else:
                assert tmP[n & 1] == n, "P V before P was written"
                assert smV[n & 1] == n, "P V before its V landed"
                done_PV.add(n)
                B["pv"].arrive()

    def tma_step():
        if tma and rng.random() < 0.3:
            bar, buf, kind, n = tma.pop(rng.randrange(len(tma)))
            if kind == "K":
                assert n < 2 or (n - 2) in done_S, "K overwritten before its S"
                smK[buf] = n
            elif kind == "V":
                assert n < 2 or (n - 2) in done_PV, "V overwritten before its P V"
                smV[buf] = n
            B[bar].arrive()

    gi, gs = issuer(), [softmax() for _ in range(n_softmax)]
    ri, rs = next(gi), [next(g) for g in gs]
    for _ in range(10 ** 6):
        if ri == "sync" and all(r == "sync" for r in rs):
            try:
                ri, rs = next(gi), [next(g) for g in gs]
            except StopIteration:
                return
            continue
        c = rng.random()
        if c < 0.3 and ri != "sync":
            ri = next(gi)
        elif c < 0.6:
            w = rng.randrange(n_softmax)
            if rs[w] != "sync":
                rs[w] = next(gs[w])
        else:
            mma_step()
            tma_step()
    raise AssertionError("deadlock")


def _items(seed):
    rng = random.Random(seed)
    return [rng.choice([0, 1, 2, 3, 4, 5, 16]) for _ in range(rng.randint(1, 8))]


@pytest.mark.parametrize("split_pfull", [True, False])
def test_forward_protocol_holds_under_random_schedules(split_pfull):
    # the kernel splits the P-written barrier per buffer; with the in-order
    # P V waits a single barrier holds as well
    for seed in range(1500):
        _simulate(_items(seed), seed, split_pfull=split_pfull)


@pytest.mark.parametrize("variant", [dict(in_order_pv=False), dict(in_order_pv=False, split_pfull=False)])
def test_protocol_variants_that_break_are_caught(variant):
    with pytest.raises(AssertionError):
        for seed in range(1500):
            _simulate(_items(seed), seed, **variant)
