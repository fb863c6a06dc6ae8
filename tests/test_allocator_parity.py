"""The library's C++ block allocator (C ABI, host code) against the oracle's
model: after every operation of scripted and random streams, identical block
tables, lengths, reference counts, free/used/cached counts, copy-on-write
pairs and failures.  Integer work: compared exactly.  No GPU needed."""
import random

import numpy as np
import pytest

import paged_kv_cache_kvc_gb300 as kvc
from oracle.allocator import AliasError, BlockAllocator, OutOfBlocks


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import os
    if not os.path.exists(kvc.LIB_PATH):
        from paged_kv_cache_kvc_gb300 import build
        build.build()
    kvc.load()


class Pair:
    """Apply each operation to both allocators and compare the outcomes."""

    def __init__(self, N, bs, free_order=None, retain=False):
        self.p = kvc.Allocator(N, bs, free_order=free_order, retain_cached=retain)
        self.o = BlockAllocator(N, bs, free_order=free_order, retain_cached=retain)
        self.N = N

    def _both(self, fp, fo):
        rp = ro = ep = eo = None
        try:
            rp = fp()
        except kvc.KvcError as e:
            ep = e.status
        try:
            ro = fo()
        except OutOfBlocks:
            eo = kvc.KVC_ERR_OOM
        except AliasError:
            eo = kvc.KVC_ERR_ALIAS
        except ValueError:
            eo = kvc.KVC_ERR_ARG
        assert (ep, rp) == (eo, ro), ((ep, rp), (eo, ro))
        return rp

    def new_seq(self):
        return self._both(self.p.new_seq, self.o.new_seq)

    def fork(self, s, n):
        return self._both(lambda: self.p.fork(s, n), lambda: self.o.fork(s, n))

    def reserve(self, s, n):
        return self._both(lambda: self.p.reserve(s, n), lambda: self.o.reserve(s, n))

    def commit(self, s, n):
        return self._both(lambda: self.p.commit(s, n), lambda: self.o.commit(s, n))

    def release(self, s):
        return self._both(lambda: self.p.release(s), lambda: self.o.release(s))

    def publish(self, s, toks, salt=0):
        return self._both(lambda: self.p.publish(s, toks, salt), lambda: self.o.publish(s, toks, salt))

    def match(self, toks, salt=0):
        return self._both(lambda: self.p.match(toks, salt), lambda: self.o.match(toks, salt))

    def lease(self, s):
        """Stamps of both sides (compared through check(), not by value)."""
        return (self.p.lease(s), self.o.lease(s))

    def check_lease(self, s, stamps):
        return self._both(lambda: self.p.check(s, stamps[0]), lambda: self.o.check(s, stamps[1]))

    def check(self, live):
        assert self.p.counts() == self.o.counts()
        assert [self.p.refcount(b) for b in range(self.N)] == self.o.ref
        if live:
            mb = max(1, max(len(self.o.seqs[s]["blocks"]) for s in live))
            table, lens = self.p.block_tables(live, mb)
            for i, s in enumerate(live):
                assert list(table[i]) == self.o.table(s, mb)
                assert lens[i] == self.o.seqs[s]["len"]


def test_table_21_1_through_both():
    x = Pair(10, 4, free_order=[7, 2, 9, 5, 0, 1, 3, 4, 6, 8])
    A = x.new_seq()
    x.reserve(A, 6)
    x.commit(A, 6)
    B = x.new_seq()
    x.reserve(B, 4)
    x.commit(B, 4)
    x.reserve(A, 3)
    x.commit(A, 3)
    C = x.fork(A, 4)
    x.check([A, B, C])
    assert x.p.refcount(7) == 2 and list(x.p.block_tables([A], 3)[0][0]) == [7, 2, 5]
    x.release(A)
    x.check([B, C])
    x.release(C)
    x.check([B])
    assert x.p.counts() == {"free": 9, "used": 1, "cached": 0}


def test_pool_exhaustion_and_reclaim_through_both():
    x = Pair(64, 4, retain=True)
    seqs = []
    for r in range(4):
        s = x.new_seq()
        x.reserve(s, 40)
        x.commit(s, 40)
        x.publish(s, [r * 100 + t for t in range(40)], salt=r)
        seqs.append(s)
    x.release(seqs.pop(0))
    x.check(seqs)
    s = x.new_seq()
    x.reserve(s, 60)              # takes the 24 free blocks, then reclaims cached ones
    x.check(seqs + [s])
    t = x.new_seq()
    x.reserve(t, 100)             # fails in both, nothing changes
    x.check(seqs + [s, t])


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("retain", [False, True])
def test_random_streams(seed, retain):
    rng = random.Random(seed)
    N, bs = rng.choice([(24, 4), (64, 16), (40, 8)])
    order = list(range(N))
    rng.shuffle(order)
    x = Pair(N, bs, free_order=order, retain=retain)
    live = []
    leases = []                                   # (id, stamps) taken along the way, checked later
    prefixes = [[rng.randrange(50) for _ in range(120)] for _ in range(3)]
    for step in range(1500):
        if live and rng.random() < 0.1:
            s = rng.choice(live)
            leases.append((s, x.lease(s)))
        for s, st in leases[-8:]:                  # stale after a release, an id reuse or copy-on-write
            x.check_lease(s, st)
        op = rng.random()
        if op < 0.15 or not live:
            live.append(x.new_seq())
        elif op < 0.5:
            s = rng.choice(live)
            n = rng.randint(0, 2 * bs + 1)
            x.reserve(s, n)
            x.commit(s, n) if rng.random() < 0.95 else None
        elif op < 0.58:
            s = rng.choice(live)
            x.commit(s, rng.randint(0, 3))       # may hit a shared block (ALIAS) or exceed capacity (ARG)
        elif op < 0.66:
            s = rng.choice(live)
            live.append(x.fork(s, rng.randint(0, x.o.seqs[s]["len"])))
        elif op < 0.76:
            s = rng.choice(live)
            p = rng.choice(prefixes)
            n = min(x.o.seqs[s]["len"], len(p))
            x.publish(s, p[:n], salt=rng.randint(0, 1))
        elif op < 0.86:
            p = rng.choice(prefixes)
            sid, hit = x.match(p[:rng.randint(0, len(p))], salt=rng.randint(0, 1))
            live.append(sid)
        else:
            s = rng.choice(live)
            x.release(s)
            live.remove(s)
        x.check(live)
