"""Plain Python block manager with prefix caching and copy-on-write
(TEST INFRASTRUCTURE ONLY).

The oracle for the native block manager of the CUDA library and for the
device block copy. Only the test suite and ``bench.py``'s CPU legs use it;
it shares no code with the library.

It is written from the rules that "LLM 推理底层：KV Cache 显存几何、GQA/MLA
压缩与 PagedAttention 调度" states in section "Prefix Caching 与
Copy-on-Write" (and the vLLM interview page, 考点 4–5), one method per rule:

  R1  identity of a full block: the chained hash
          H_k = Hash(H_{k-1}, token ids of block k),   H_{-1} = 0
      so a block's hash names its whole prefix (``chain_hashes``);
  R2  reuse: a prompt's full blocks are looked up by H_0, H_1, ... in order;
      the lookups stop at the first miss, every hit is shared (one more
      reference) and its tokens count as cached (``_cached_prefix``);
  R3  release without wiping: a block nobody references keeps its contents
      and hash and waits in a least-recently-released order; a new block is
      the one released longest ago, and only then does it lose its old hash
      (``_release``, ``_claim``, ``_recycle``);
  R4  sharing by reference: forking a sequence (beam search, parallel
      sampling) adds one reference to each of its blocks (``fork``);
  R5  copy-on-write: a token appended to a last block that is partly filled
      and shared goes to a private copy of that block; the others keep the
      original (``append_slot``); a full last block (or none) gets a new one.

Readings where the pages leave a step open:
  * Hash = BLAKE2b with an 8-byte digest over ``hash_input`` (the parent as
    8 little-endian bytes, then each token id as 4 little-endian bytes); the
    digest read as a little-endian integer. Token ids are >= 0.
  * Only prompt blocks get a hash; appended tokens never create one.
  * A hash names at most one block: a block registered under a hash that an
    older block still carries takes the hash over. (With blocks released in
    table order and recycled oldest first, the older copies of a prefix are
    recycled before the new blocks are registered, so this does not arise
    through these calls; the rule keeps the map exact regardless.)
  * Every method either succeeds or raises MemoryError and changes nothing.
    A prompt is planned in full first (hits, then the number of blocks it
    must recycle, counting that hit blocks waiting in the pool are no longer
    free); a half-admitted prompt could not simply be freed, its new blocks
    would carry hashes of K/V that is never written.
  * Blocks start out free in id order (block 0 is recycled first).
  * ``append_slot`` returns the new token's slot (block * 16 + offset) and
    the (source, destination) pair the caller must copy on the device, or
    None.
"""
from __future__ import annotations

import hashlib
import heapq
from typing import Dict, List, Optional, Tuple

import numpy as np


# ------------------------------------------------------------------- R1
def hash_input(parent: int, tokens) -> bytes:
    """The bytes a block hash digests: parent (8 bytes LE), then each token
    id (4 bytes LE)."""
    out = bytearray(int(parent).to_bytes(8, "little"))
    for t in tokens:
        out += int(t).to_bytes(4, "little")
    return bytes(out)


def block_hash(parent: int, tokens) -> int:
    """H_k from H_{k-1} (`parent`) and the token ids of block k."""
    return int.from_bytes(hashlib.blake2b(hash_input(parent, tokens), digest_size=8).digest(),
                          "little")


def chain_hashes(token_ids, block_size: int) -> List[int]:
    """H_0, H_1, ... of every full block of a token sequence."""
    hashes: List[int] = []
    parent = 0
    for k in range(len(token_ids) // block_size):
        parent = block_hash(parent, token_ids[k * block_size:(k + 1) * block_size])
        hashes.append(parent)
    return hashes


class BlockState:
    """One physical block: holders, prefix hash (full prompt blocks only),
    and the token ids written into its slots."""

    __slots__ = ("ref", "hash", "tokens")

    def __init__(self):
        self.ref = 0
        self.hash: Optional[int] = None
        self.tokens: List[int] = []


class Allocator:
    def __init__(self, num_blocks: int, block_size: int = 16):
        self.block_size = block_size
        self.blocks = [BlockState() for _ in range(num_blocks)]
        self.by_hash: Dict[int, int] = {}
        # R3: free blocks ordered by release time. A min-heap of (stamp, id);
        # a block's live stamp is _stamp[id] (None while held), entries with
        # another stamp are stale and skipped.
        self._stamp: List[Optional[int]] = list(range(num_blocks))
        self._heap: List[Tuple[int, int]] = [(i, i) for i in range(num_blocks)]
        self._clock = num_blocks
        self._free = num_blocks

    # ---------------------------------------------------------------- R3
    def _release(self, bid: int) -> None:
        blk = self.blocks[bid]
        if blk.ref <= 0:
            raise ValueError(f"block {bid} is not held")
        blk.ref -= 1
        if blk.ref == 0:
            self._stamp[bid] = self._clock
            heapq.heappush(self._heap, (self._clock, bid))
            self._clock += 1
            self._free += 1

    def _claim(self, bid: int) -> None:
        """One more holder; a free block leaves the free order."""
        if self._stamp[bid] is not None:
            self._stamp[bid] = None
            self._free -= 1
        self.blocks[bid].ref += 1

    def _recycle(self, tokens: List[int]) -> int:
        """The block released longest ago, stripped of its old identity and
        given `tokens`, with one holder."""
        while True:
            if not self._heap:
                raise MemoryError("no free KV cache block")
            stamp, bid = heapq.heappop(self._heap)
            if self._stamp[bid] == stamp:
                break
        self._claim(bid)
        blk = self.blocks[bid]
        if blk.hash is not None:
            del self.by_hash[blk.hash]
            blk.hash = None
        blk.tokens = list(tokens)
        return bid

    # ---------------------------------------------------------------- R2
    def _cached_prefix(self, hashes: List[int]) -> List[int]:
        """Block ids of the leading hashes found in the cache (up to the
        first miss)."""
        hits: List[int] = []
        for h in hashes:
            bid = self.by_hash.get(h)
            if bid is None:
                break
            hits.append(bid)
        return hits

    def allocate_for_prompt(self, token_ids) -> Tuple[List[int], int]:
        """Blocks for a whole prompt: the cached prefix shared, the rest
        recycled (full ones registered under their hash). Returns (table,
        number of cached tokens)."""
        bs = self.block_size
        ids = [int(t) for t in token_ids]
        hashes = chain_hashes(ids, bs)
        hits = self._cached_prefix(hashes)
        n_blocks = -(-len(ids) // bs)
        waiting_hits = sum(1 for bid in hits if self.blocks[bid].ref == 0)
        if n_blocks - len(hits) > self._free - waiting_hits:
            raise MemoryError("no free KV cache block")
        table = []
        for bid in hits:
            self._claim(bid)
            table.append(bid)
        for k in range(len(hits), n_blocks):
            bid = self._recycle(ids[k * bs:(k + 1) * bs])
            if k < len(hashes):
                older = self.by_hash.get(hashes[k])
                if older is not None:           # one block per hash
                    self.blocks[older].hash = None
                self.blocks[bid].hash = hashes[k]
                self.by_hash[hashes[k]] = bid
            table.append(bid)
        return table, len(hits) * bs

    # ---------------------------------------------------------------- R5
    def append_slot(self, table: List[int], token: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Write one decoded token at the end of a sequence (its table is
        updated in place). Returns (slot, copy pair or None)."""
        bs = self.block_size
        tail = self.blocks[table[-1]] if table else None
        if tail is None or len(tail.tokens) == bs:          # no room: a new block
            bid = self._recycle([int(token)])
            table.append(bid)
            return bid * bs, None
        if tail.ref == 1:                                   # private: write in place
            tail.tokens.append(int(token))
            return table[-1] * bs + len(tail.tokens) - 1, None
        src = table[-1]                                     # shared: copy, then write
        bid = self._recycle(tail.tokens + [int(token)])
        self._release(src)
        table[-1] = bid
        return bid * bs + len(self.blocks[bid].tokens) - 1, (src, bid)

    # ---------------------------------------------------------------- R4
    def fork(self, table: List[int]) -> List[int]:
        for bid in table:
            self._claim(bid)
        return list(table)

    def free_sequence(self, table: List[int]) -> None:
        for bid in table:
            if self.blocks[bid].ref <= 0:
                raise ValueError(f"block {bid} is not held")
        for bid in table:
            self._release(bid)

    # ------------------------------------------------------- introspection
    def ref_count(self, bid: int) -> int:
        return self.blocks[bid].ref

    def hash_of(self, bid: int) -> Optional[int]:
        return self.blocks[bid].hash

    def num_tokens(self, bid: int) -> int:
        return len(self.blocks[bid].tokens)

    def free_order(self) -> List[int]:
        """Free blocks, the next one to be recycled first."""
        return [bid for _, bid in sorted((s, b) for b, s in enumerate(self._stamp)
                                         if s is not None)]

    def num_free(self) -> int:
        return self._free


def block_copy(k_cache: np.ndarray, v_cache: np.ndarray, pairs,
               k_scale: Optional[np.ndarray] = None, v_scale: Optional[np.ndarray] = None):
    """The device half of copy-on-write: for every (src, dst) pair, block dst
    of each array (indexed by block first) becomes a copy of block src, all
    heads and all slots. Destinations are distinct and none is a source."""
    arrays = [a for a in (k_cache, v_cache, k_scale, v_scale) if a is not None]
    for src, dst in pairs:
        for a in arrays:
            a[dst] = a[src]
