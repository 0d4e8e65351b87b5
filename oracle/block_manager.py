"""Reference model of the prefix-caching block manager -- TEST INFRASTRUCTURE ONLY.

Only the tests and ``__graft_entry__.smoke()`` may use it; the library's own
manager (C++) shares no code with it.

What it models: the paged KV pool of 16-token blocks reached through per-
sequence block tables ("LLM Inference Server", Optional Bonus Extensions:
Paged KV-Cache Block Allocator; "LLM Inference Server From Scratch", How it
works, 3 Block Manager), with the hash-keyed prefix cache of "LLM Inference
Server", Stage 1 (prefilled KV of a common system prompt stored once and
reused by later requests, with hit/miss tracking) and the block sharing across
requests of "Mini inference engine", step 2 (stretch).  The pages fix none of
the policies; every one below is a plain, deterministic choice, so that two
implementations of the same rules must agree on every block id:

* a full block is keyed by FNV-1a (64-bit) over the little-endian bytes of
  its parent's key (0 for the first block) followed by its 16 token ids; a
  cache hit also compares the stored parent key and tokens;
* a new prompt reuses its cached full blocks from the start until the first
  miss (hits / misses count full prompt blocks), then allocates the rest; its
  newly allocated full blocks are entered in the cache at once (unless the key
  is already taken);
* an append that opens a block allocates one; an append into a last block
  that another table also holds copies it first (copy-on-write: the pair
  (source, new block) is reported for the caller to copy on the GPU); a block
  that fills up is entered in the cache;
* freeing a sequence releases its blocks last to first; a released block that
  is in the cache waits, unreferenced, on a least-recently-released list,
  others return to the free set;
* allocation takes the lowest free block id, else evicts the least recently
  released cached block (removing its key); with neither it fails and changes
  nothing.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Tuple

BLOCK = 16
FNV_OFFSET = 0xCBF29CE484222325
FNV_PRIME = 0x100000001B3
MASK64 = (1 << 64) - 1


def fnv1a64(data: bytes) -> int:
    h = FNV_OFFSET
    for b in data:
        h ^= b
        h = (h * FNV_PRIME) & MASK64
    return h


def block_key(parent: int, tokens: List[int]) -> int:
    data = parent.to_bytes(8, "little")
    for t in tokens:
        data += (t & 0xFFFFFFFF).to_bytes(4, "little")
    return fnv1a64(data)


class NoBlocks(Exception):
    pass


class BlockManagerRef:
    def __init__(self, num_blocks: int, max_blocks_per_seq: int, max_seqs: int):
        self.nb = num_blocks
        self.max_blocks = max_blocks_per_seq
        self.max_seqs = max_seqs
        self.ref = [0] * num_blocks
        self.key: List[Optional[Tuple[int, int, Tuple[int, ...]]]] = [None] * num_blocks  # (key, parent, tokens)
        self.free = set(range(num_blocks))
        self.lru: Dict[int, int] = {}          # cached, unreferenced block -> release tick
        self.cache: Dict[int, int] = {}        # key -> block
        self.tick = 0
        self.seqs: Dict[int, dict] = {}
        self.stats = {"hit_blocks": 0, "miss_blocks": 0, "cow_copies": 0, "evictions": 0}

    # ---- allocation ---------------------------------------------------------
    def _available(self) -> int:
        return len(self.free) + len(self.lru)

    def _alloc(self) -> int:
        if self.free:
            b = min(self.free)
            self.free.remove(b)
        elif self.lru:
            b = min(self.lru, key=lambda x: (self.lru[x], x))
            del self.lru[b]
            k = self.key[b]
            if k is not None and self.cache.get(k[0]) == b:
                del self.cache[k[0]]
            self.key[b] = None
            self.stats["evictions"] += 1
        else:
            raise NoBlocks()
        self.ref[b] = 1
        return b

    def _register(self, b: int, parent: int, tokens: List[int]) -> int:
        k = block_key(parent, tokens)
        if k not in self.cache:
            self.cache[k] = b
            self.key[b] = (k, parent, tuple(tokens))
        return k

    def _lookup(self, parent: int, tokens: List[int]) -> Optional[int]:
        k = block_key(parent, tokens)
        b = self.cache.get(k)
        if b is None:
            return None
        _, p, t = self.key[b]
        return b if p == parent and list(t) == list(tokens) else None

    # ---- operations -----------------------------------------------------------
    def add_sequence(self, seq: int, prompt: List[int]) -> Tuple[int, List[int]]:
        """Returns (cached prompt tokens, slots of every prompt position)."""
        if not (0 <= seq < self.max_seqs) or seq in self.seqs:
            raise ValueError("bad sequence id")
        n = len(prompt)
        if (n + BLOCK - 1) // BLOCK > self.max_blocks:
            raise ValueError("prompt longer than the block table")
        full = n // BLOCK
        hits = []
        parent = 0
        for i in range(full):
            b = self._lookup(parent, prompt[i * BLOCK:(i + 1) * BLOCK])
            if b is None:
                break
            hits.append(b)
            parent = block_key(parent, prompt[i * BLOCK:(i + 1) * BLOCK])
        need = (n + BLOCK - 1) // BLOCK - len(hits)
        # hit blocks waiting on the LRU list are taken out of it, so they do not count as available
        if self._available() - sum(1 for b in hits if b in self.lru) < need:
            raise NoBlocks()
        table = []
        for b in hits:
            if b in self.lru:
                del self.lru[b]
            self.ref[b] += 1
            table.append(b)
        self.stats["hit_blocks"] += len(hits)
        self.stats["miss_blocks"] += full - len(hits)
        for i in range(len(hits), (n + BLOCK - 1) // BLOCK):
            b = self._alloc()
            table.append(b)
            toks = prompt[i * BLOCK:(i + 1) * BLOCK]
            if len(toks) == BLOCK:
                parent = self._register(b, parent, toks)
        tail = list(prompt[full * BLOCK:])
        self.seqs[seq] = {"table": table, "len": n, "tail": tail, "parent": parent}
        slots = [table[p // BLOCK] * BLOCK + p % BLOCK for p in range(n)]
        return len(hits) * BLOCK, slots

    def append(self, seq: int, tokens: List[int]) -> Tuple[List[int], List[Tuple[int, int]]]:
        """Returns (slots of the new tokens, copy-on-write pairs (src, dst))."""
        s = self.seqs[seq]
        n0 = s["len"]
        if (n0 + len(tokens) + BLOCK - 1) // BLOCK > self.max_blocks:
            raise ValueError("sequence longer than the block table")
        opens = sum(1 for p in range(n0, n0 + len(tokens)) if p % BLOCK == 0)
        cow = 1 if (tokens and n0 % BLOCK != 0 and self.ref[s["table"][-1]] > 1) else 0
        if self._available() < opens + cow:
            raise NoBlocks()
        slots, copies = [], []
        for tok in tokens:
            p = s["len"]
            if p % BLOCK == 0:
                s["table"].append(self._alloc())
                s["tail"] = []
            else:
                last = s["table"][-1]
                if self.ref[last] > 1:
                    nb = self._alloc()
                    copies.append((last, nb))
                    self.ref[last] -= 1
                    s["table"][-1] = nb
                    self.stats["cow_copies"] += 1
            slots.append(s["table"][-1] * BLOCK + p % BLOCK)
            s["tail"].append(tok)
            s["len"] = p + 1
            if s["len"] % BLOCK == 0:
                s["parent"] = self._register(s["table"][-1], s["parent"], s["tail"])
                s["tail"] = []
        return slots, copies

    def append_step(self, seqs: List[int], tokens: List[int]):
        """One token for each listed sequence (in order), all or nothing:
        returns (slots, copy-on-write pairs in call order)."""
        need, dec = 0, {}
        for sq in seqs:
            s = self.seqs[sq]
            if (s["len"] + 1 + BLOCK - 1) // BLOCK > self.max_blocks:
                raise ValueError("sequence longer than the block table")
            if s["len"] % BLOCK == 0:
                need += 1
            else:
                last = s["table"][-1]
                if self.ref[last] - dec.get(last, 0) > 1:
                    need += 1
                    dec[last] = dec.get(last, 0) + 1
        if len(set(seqs)) != len(seqs):
            raise ValueError("a sequence listed twice")
        if self._available() < need:
            raise NoBlocks()
        slots, copies = [], []
        for sq, tok in zip(seqs, tokens):
            sl, cp = self.append(sq, [tok])
            slots += sl
            copies += cp
        return slots, copies

    def fork(self, parent: int, child: int):
        if child in self.seqs or not (0 <= child < self.max_seqs):
            raise ValueError("bad child id")
        p = self.seqs[parent]
        for b in p["table"]:
            self.ref[b] += 1
        self.seqs[child] = {"table": list(p["table"]), "len": p["len"], "tail": list(p["tail"]),
                            "parent": p["parent"]}

    def free_sequence(self, seq: int):
        s = self.seqs.pop(seq)
        for b in reversed(s["table"]):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                if self.key[b] is not None and self.cache.get(self.key[b][0]) == b:
                    self.tick += 1
                    self.lru[b] = self.tick
                else:
                    self.key[b] = None
                    self.free.add(b)

    def table(self, seq: int) -> List[int]:
        return list(self.seqs[seq]["table"])

    def length(self, seq: int) -> int:
        return self.seqs[seq]["len"]

    def counts(self) -> dict:
        d = dict(self.stats)
        d.update(free_blocks=len(self.free), cached_free_blocks=len(self.lru),
                 used_blocks=sum(1 for r in self.ref if r > 0))
        return d
