"""Pins of the oracle's block-allocator model to what the pages state (no GPU).

- Table 21.1 and its steps 1-5 ("KV cache: Generation state, latency, and
  allocation" 21.5): which blocks are taken, shared, kept and freed.
- "KV Cache Explained", "Follow the 32 GiB pool until it cannot allocate one
  more block": the 16 384-block pool, free blocks first, then reclaiming idle
  cached prefixes, then failure once everything is pinned.
- Same page, "Prefix reuse saves prefill": 6 GiB separate vs 4 GiB shared.
- xf_kv_cache page, "End-to-end flow": the 75-block shared prefix at
  refcount 40, private blocks for the new tokens, release on completion.
"""
import pytest

from oracle.allocator import AliasError, BlockAllocator, OutOfBlocks

MIB2 = 2          # one 16-token block of the Llama-style shape is 2 MiB across the layers


def test_table_21_1_steps_1_to_5():
    # blocks of four positions; the page's chosen ids 7, 2 (A), 9 (B), then 5 (A's third block)
    a = BlockAllocator(10, 4, free_order=[7, 2, 9, 5, 0, 1, 3, 4, 6, 8])
    A = a.new_seq()
    a.reserve(A, 6)
    a.commit(A, 6)
    B = a.new_seq()
    a.reserve(B, 4)
    a.commit(B, 4)
    assert a.table(A, 3) == [7, 2, -1] and a.table(B, 3) == [9, -1, -1]
    # step 1: positions 6 and 7 fill block 2, no new block
    assert a.reserve(A, 2) == [] and a.table(A, 3) == [7, 2, -1]
    a.commit(A, 2)
    # step 2: position 8 needs logical block 2; the allocator maps free block 5
    assert a.reserve(A, 1) == [] and a.table(A, 3) == [7, 2, 5]
    a.commit(A, 1)
    # step 3: C shares A's complete first block 7; reference count 2
    C = a.fork(A, 4)
    assert a.table(C, 3) == [7, -1, -1] and a.ref[7] == 2
    # step 4: A finishes; 2 and 5 return to the free pool, 7 stays live for C, B still owns 9
    a.release(A)
    assert a.ref[7] == 1 and a.ref[2] == 0 and a.ref[5] == 0 and a.ref[9] == 1
    assert 2 in a.free and 5 in a.free and 7 not in a.free and 9 not in a.free
    # step 5: C finishes; 7 becomes free under the immediate-release policy; B's release frees 9
    a.release(C)
    assert a.ref[7] == 0 and 7 in a.free
    a.release(B)
    assert sorted(a.free) == list(range(10))


def test_table_21_1_step_5_retention_keeps_an_evictable_entry():
    a = BlockAllocator(10, 4, free_order=[7, 2, 9, 5, 0, 1, 3, 4, 6, 8], retain_cached=True)
    A = a.new_seq()
    a.reserve(A, 9)
    a.commit(A, 9)
    toks = list(range(100, 109))
    a.publish(A, toks)                       # full blocks 7 and 2 get identities
    C = a.fork(A, 4)
    a.release(A)
    assert 5 in a.free and 2 in a.cached      # 2 was full and published: kept as evictable
    a.release(C)
    assert 7 in a.cached and a.ref[7] == 0
    D, hit = a.match(toks)                   # the retained prefix is found again
    assert hit == 8 and a.table(D, 2) == [7, 2] and a.ref[7] == 1 and not a.cached


def test_32_gib_pool_until_one_more_block_fails():
    N = 16384                                  # 32 GiB / 2 MiB
    assert N * MIB2 == 32 * 1024
    a = BlockAllocator(N, 16, retain_cached=True)
    running = []
    for r in range(6):                         # six requests hold 24 GiB of active KV
        s = a.new_seq()
        a.reserve(s, 32768)
        a.commit(s, 32768)
        running.append(s)
    for r in range(3):                         # 6 GiB of completed prefixes kept for reuse (3 x 2 GiB)
        s = a.new_seq()
        a.reserve(s, 16384)
        a.commit(s, 16384)
        a.publish(s, [r * 1_000_000 + t for t in range(16384)], salt=r)
        a.release(s)
    c = a.counts()
    assert c["used"] * MIB2 == 24 * 1024 and c["cached"] * MIB2 == 6 * 1024 and c["free"] * MIB2 == 2 * 1024
    # a 32 768-token prompt needs 4 GiB: the 2 GiB free plus 2 GiB reclaimed from idle cached prefixes
    new = a.new_seq()
    a.reserve(new, 32768)
    assert a.counts()["free"] == 0 and a.counts()["cached"] * MIB2 == 4 * 1024
    assert all(len(a.seqs[s]["blocks"]) == 2048 for s in running)      # none of the six had to stop
    # the running requests grow by another 4 GiB: the rest of the idle cache is reclaimed
    for s in running[:4]:
        a.reserve(s, 8192)
        a.commit(s, 8192)
    assert a.counts() == {"free": 0, "used": N, "cached": 0}
    # now every block is referenced by active work: one more block cannot be provided
    s = a.new_seq()
    with pytest.raises(OutOfBlocks):
        a.reserve(s, 1)
    assert a.counts() == {"free": 0, "used": N, "cached": 0}       # and nothing changed


def test_prefix_sharing_6_vs_4_gib():
    a = BlockAllocator(4096, 16)
    toks = list(range(24576))
    s1 = a.new_seq()
    a.reserve(s1, 24576)
    a.commit(s1, 24576)
    a.publish(s1, toks)
    s2, hit = a.match(toks[:16384])          # the second request shares the first 16 384 tokens
    assert hit == 16384
    a.reserve(s2, 8192)
    a.commit(s2, 8192)
    unique = a.counts()["used"]
    assert unique * MIB2 == 4 * 1024                       # one physical prefix + two 8 192-token suffixes
    separate = 2 * 24576 // 16
    assert separate * MIB2 == 6 * 1024


def test_end_to_end_flow_refcount_40():
    a = BlockAllocator(20000, 16, retain_cached=True)
    prefix = [7_000 + t for t in range(1200)]
    owner = a.new_seq()
    a.reserve(owner, 1200)
    a.commit(owner, 1200)
    a.publish(owner, prefix)
    others = [a.match(prefix)[0] for _ in range(39)]
    shared = a.table(owner, 75)
    assert all(a.ref[b] == 40 for b in shared)           # "first 75 blocks already resident with refcount 40"
    convo = prefix + [9_000 + t for t in range(600)]     # a 1 800-token conversation
    seq, hit = a.match(convo)
    assert hit == 1200 and a.table(seq, 75) == shared and all(a.ref[b] == 41 for b in shared)
    free0 = a.counts()["free"]
    a.reserve(seq, 600)                                   # blocks only for the 600 unshared tokens
    a.commit(seq, 600)
    assert free0 - a.counts()["free"] == 113 - 75
    for t in range(900):                                  # decode: a fresh block every 16 tokens
        before = len(a.seqs[seq]["blocks"])
        a.reserve(seq, 1)
        a.commit(seq, 1)
        assert len(a.seqs[seq]["blocks"]) - before == (1 if (1800 + t) % 16 == 0 else 0)
    private = a.seqs[seq]["blocks"][75:]
    assert len(private) == -(-2700 // 16) - 75
    a.release(seq)                                         # private blocks return, shared ones decrement
    assert all(b in a.free for b in private) and all(a.ref[b] == 40 for b in shared)
    for s in others:
        a.release(s)


def test_copy_on_write_of_a_shared_partial_block():
    a = BlockAllocator(8, 4)
    A = a.new_seq()
    a.reserve(A, 6)
    a.commit(A, 6)                            # blocks 0, 1; block 1 holds 2 of 4 positions
    B = a.fork(A, 6)                          # shares both, including the partly filled one
    assert a.ref[1] == 2
    with pytest.raises(AliasError):
        a.commit(B, 1)                         # writing without a reserve would change A's view
    pairs = a.reserve(B, 1)                   # B's next write lands in shared block 1: copy it first
    assert pairs == [(1, 2)] and a.table(B, 2) == [0, 2] and a.ref[1] == 1 and a.ref[2] == 1
    a.commit(B, 1)
    assert a.reserve(A, 1) == [] and a.table(A, 2) == [0, 1]     # A's block is private again
    C = a.fork(A, 4)                          # sharing a full block only: no copy on the next write
    assert a.reserve(C, 3) == [] and a.table(C, 2) == [0, 3]


def test_invariants_under_random_operations():
    import random
    rng = random.Random(5)
    a = BlockAllocator(40, 4, retain_cached=True)
    live = []
    for step in range(3000):
        op = rng.random()
        try:
            if op < 0.2 or not live:
                live.append(a.new_seq())
            elif op < 0.55:
                s = rng.choice(live)
                n = rng.randint(1, 9)
                a.reserve(s, n)
                a.commit(s, n)
            elif op < 0.65:
                s = rng.choice(live)
                live.append(a.fork(s, rng.randint(0, a.seqs[s]["len"])))
            elif op < 0.75:
                s = rng.choice(live)
                a.publish(s, [t % 5 for t in range(a.seqs[s]["len"])])
            elif op < 0.85:
                live.append(a.match([t % 5 for t in range(rng.randint(0, 30))])[0])
            else:
                s = rng.choice(live)
                a.release(s)
                live.remove(s)
        except OutOfBlocks:
            pass
        refs = [0] * a.N
        for s in live:
            for b in a.seqs[s]["blocks"]:
                refs[b] += 1
        assert refs == a.ref
        assert len(set(a.free)) + len(set(a.cached)) + sum(1 for r in refs if r) == a.N
        assert not set(a.free) & set(a.cached)


def test_lease_race_generation_check():
    """"KV Cache Explained", "The lease race when KV crosses workers": a
    receiver holds a request's table under a lease; the source releases the
    request (the lease expired) and hands the same physical blocks to another
    request; the receiver's generation check must now fail, although the block
    ids it holds are valid and mapped again.  Mapping new blocks at the end of a
    table keeps its stamp; copy-on-write replacing an entry does not."""
    a = BlockAllocator(4, 4, free_order=[3, 1, 0, 2])
    src = a.new_seq()
    a.reserve(src, 8)
    a.commit(src, 8)
    stamp = a.lease(src)
    table = a.table(src, 2)
    assert table == [3, 1] and a.check(src, stamp)
    a.reserve(src, 4)                 # grows into a third block: the first two entries are unchanged
    a.commit(src, 4)
    assert a.check(src, stamp) and a.table(src, 3)[:2] == table
    a.release(src)                    # the lease expires at the source
    assert not a.check(src, stamp)
    other = a.new_seq()               # the id and the blocks go to another request
    a.reserve(other, 16)
    assert other == src and sorted(a.table(other, 4)) == [0, 1, 2, 3]
    assert not a.check(src, stamp)    # same id, same block ids: still stale
    assert a.check(other, a.lease(other))
    # copy-on-write replacing an entry makes earlier stamps stale
    b = BlockAllocator(8, 4)
    x = b.new_seq()
    b.reserve(x, 6)
    b.commit(x, 6)
    y = b.fork(x, 6)
    st_y = b.lease(y)
    assert b.reserve(y, 1) == [(1, 2)]
    assert not b.check(y, st_y) and b.check(x, b.lease(x))
    with pytest.raises(ValueError):
        b.check(99, st_y)
