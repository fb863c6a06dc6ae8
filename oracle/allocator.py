"""Plain model of the paged-cache block allocator -- TEST INFRASTRUCTURE ONLY.

Follows "KV cache: Generation state, latency, and allocation" 21.5 and Table
21.1 (blocks mapped as a sequence grows; a shared block carries one reference
per mapping request; full shared blocks stay immutable and a shared, partly
filled block is copied before a write; release drops references; at count
zero a block returns to the free pool, or under a retention policy stays as an
evictable cached entry), 21.4 (a block's identity is its configuration
identity / salt plus every token id up to its end: the chain h_i =
hash(h_{i-1}, tokens_i) written out as the whole prefix), and "KV Cache
Explained", "Follow the 32 GiB pool until it cannot allocate one more block"
(free blocks first, then unreferenced cached blocks, then failure).

Written with Python lists and dicts so that it can be read against the
passages; it shares nothing with the library's C++ allocator.
"""
from __future__ import annotations

from collections import deque


class OutOfBlocks(Exception):
    pass


class AliasError(Exception):
    pass


class BlockAllocator:
    def __init__(self, num_blocks, block_size, free_order=None, retain_cached=False):
        self.N, self.bs, self.retain = num_blocks, block_size, retain_cached
        self.free = deque(range(num_blocks) if free_order is None else [int(b) for b in free_order])
        self.cached = []                 # evictable blocks, least recently released first
        self.ref = [0] * num_blocks
        self.identity = {}               # block -> identity (salt, prefix token tuple)
        self.index = {}                  # identity -> block
        self.seqs = []                   # per id: None or {"blocks": [...], "len": n, "replaced": r}
        self.handed_out = []             # per id: how many times the id was given to a new sequence

    # ---------------------------------------------------------- blocks
    def _forget(self, b):
        ident = self.identity.pop(b, None)
        if ident is not None and self.index.get(ident) == b:
            del self.index[ident]

    def _take(self):
        if self.free:
            b = self.free.popleft()
        elif self.cached:
            b = self.cached.pop(0)       # reclaim the least recently released cached block
            self._forget(b)
        else:
            raise OutOfBlocks()
        self.ref[b] = 1
        return b

    def _drop(self, b):
        self.ref[b] -= 1
        if self.ref[b] > 0:
            return
        if self.retain and b in self.identity:
            self.cached.append(b)
        else:
            self._forget(b)
            self.free.append(b)

    def _add(self, b):
        if b in self.cached:             # a prefix hit revives an evictable entry
            self.cached.remove(b)
            self.ref[b] = 0
        self.ref[b] += 1

    def available(self):
        return len(self.free) + len(self.cached)

    # ---------------------------------------------------------- sequences
    def _new_id(self):
        for i, s in enumerate(self.seqs):
            if s is None:
                self.seqs[i] = {"blocks": [], "len": 0, "replaced": 0}
                self.handed_out[i] += 1
                return i
        self.seqs.append({"blocks": [], "len": 0, "replaced": 0})
        self.handed_out.append(1)
        return len(self.seqs) - 1

    def new_seq(self):
        return self._new_id()

    def fork(self, src, n_tokens):
        s = self.seqs[src]
        if not 0 <= n_tokens <= s["len"]:
            raise ValueError("fork length outside the source sequence")
        nb = -(-n_tokens // self.bs)
        i = self._new_id()
        d = self.seqs[i]
        d["blocks"] = list(self.seqs[src]["blocks"][:nb])
        d["len"] = n_tokens
        for b in d["blocks"]:
            self._add(b)
        return i

    def reserve(self, seq, n_tokens):
        """Room for n_tokens more positions; returns [(old, new)] copy-on-write pairs."""
        s = self.seqs[seq]
        target = s["len"] + n_tokens
        need = max(0, -(-target // self.bs) - len(s["blocks"]))
        w = s["len"] // self.bs
        cow = n_tokens > 0 and s["len"] % self.bs != 0 and w < len(s["blocks"]) and self.ref[s["blocks"][w]] > 1
        if not cow and need == 0:
            return []
        if self.available() < need + (1 if cow else 0):
            raise OutOfBlocks()
        pairs = []
        if cow:
            fresh = self._take()
            old = s["blocks"][w]
            pairs.append((old, fresh))
            s["blocks"][w] = fresh
            s["replaced"] += 1           # a table handed out earlier still maps the old block
            self._drop(old)
        for _ in range(need):
            s["blocks"].append(self._take())
        return pairs

    def commit(self, seq, n_tokens):
        s = self.seqs[seq]
        if n_tokens < 0 or s["len"] + n_tokens > len(s["blocks"]) * self.bs:
            raise ValueError("commit beyond the reserved blocks")
        for t in range(s["len"], s["len"] + n_tokens):
            if self.ref[s["blocks"][t // self.bs]] > 1:
                raise AliasError()
        s["len"] += n_tokens

    def release(self, seq):
        for b in self.seqs[seq]["blocks"]:
            self._drop(b)
        self.seqs[seq] = None

    def publish(self, seq, tokens, salt=0):
        s = self.seqs[seq]
        for i in range(len(tokens) // self.bs):
            ident = (salt, tuple(int(t) for t in tokens[:(i + 1) * self.bs]))
            b = s["blocks"][i]
            if b not in self.identity and ident not in self.index:
                self.identity[b] = ident
                self.index[ident] = b

    def match(self, tokens, salt=0):
        hits = []
        for i in range(len(tokens) // self.bs):
            ident = (salt, tuple(int(t) for t in tokens[:(i + 1) * self.bs]))
            if ident not in self.index:
                break
            hits.append(self.index[ident])
        i = self._new_id()
        self.seqs[i]["blocks"] = hits
        self.seqs[i]["len"] = len(hits) * self.bs
        for b in hits:
            self._add(b)
        return i, len(hits) * self.bs

    # ---------------------------------------------------------- lease stamps
    # "KV Cache Explained", "The lease race when KV crosses workers": whoever
    # receives a request's blocks must be able to tell that the lease expired
    # (the blocks may belong to another request now) -- a generation check, a
    # mismatch counting as failure.  A stamp names the sequence id's hand-out
    # count and how many of its table entries copy-on-write has replaced.
    def lease(self, seq):
        s = self.seqs[seq]
        if s is None:
            raise ValueError("no such sequence")
        return (self.handed_out[seq], s["replaced"])

    def check(self, seq, stamp):
        """True while the stamp still describes the live sequence's table."""
        if not 0 <= seq < len(self.seqs):
            raise ValueError("id never handed out")
        return self.seqs[seq] is not None and self.lease(seq) == stamp

    # ---------------------------------------------------------- views
    def table(self, seq, max_blocks):
        bl = self.seqs[seq]["blocks"]
        return bl + [-1] * (max_blocks - len(bl))

    def counts(self):
        return {"free": len(self.free), "used": self.N - len(self.free) - len(self.cached), "cached": len(self.cached)}
