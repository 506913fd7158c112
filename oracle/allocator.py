"""Plain Python block allocator with chained-hash prefix caching and
copy-on-write (TEST INFRASTRUCTURE ONLY).

This is the oracle for the native allocator in the CUDA library and for the
device block copy. Only the test suite and ``bench.py``'s CPU legs use it; it
shares no code with the library.

What it follows ("LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度",
section "Prefix Caching 与 Copy-on-Write" and its allocator reference):
  * a full block k of a prompt is named by the chained hash
        H_k = Hash(H_{k-1}, tokens of block k),   H_{-1} = 0,
    with Hash = BLAKE2b, 8-byte digest, over the parent as 8 little-endian
    bytes followed by each token id as 4 little-endian bytes;
  * a block whose reference count drops to zero is not wiped: it joins an
    LRU pool of evictable blocks and stays findable by its hash until it is
    taken for new data (then its hash is dropped);
  * a new prompt matches H_0, H_1, ... in order; every hit increments the
    block's reference count and counts 16 tokens as cached; the first miss
    ends matching for the rest of the prompt;
  * appending a decoded token to a last block that is full takes a new block;
    appending to a last block that is not full but shared (reference count
    > 1) copies it to a new block first (copy-on-write) and leaves the shared
    block to the other holders.
Forking a table for beam search or parallel sampling increments the
reference count of each of its blocks (same page, 考点 4: branches point at
the same physical blocks and each holder counts once).

Readings where the pages leave a step open:
  * every method either succeeds or raises MemoryError and leaves the
    allocator exactly as it was. A prompt first counts its hits (matching
    changes nothing) and the blocks it must take; if the pool, less the hit
    blocks that sit in it, is too small, it fails before any change (a
    half-done prompt cannot be released like a sequence: its new blocks
    already carry hashes of KV data that will never be written).
    ``append_slot`` takes the new block before it touches any reference
    count;
  * appending to an empty table takes a new block;
  * ``append_slot`` returns the slot of the new token (block * 16 + offset)
    and the (source, destination) pair that the caller must copy on the
    device, or None;
  * only prompt blocks get a hash (the reference hashes nothing on append).
"""
from __future__ import annotations

import hashlib
from collections import OrderedDict
from typing import List, Optional, Tuple

import numpy as np


def block_hash(parent: int, tokens) -> int:
    """H_k = BLAKE2b-64(parent as 8 LE bytes || each token as 4 LE bytes)."""
    h = hashlib.blake2b(digest_size=8)
    h.update(int(parent).to_bytes(8, "little", signed=False))
    for t in tokens:
        h.update(int(t).to_bytes(4, "little", signed=False))
    return int.from_bytes(h.digest(), "little", signed=False)


class _Block:
    __slots__ = ("ref", "hash", "tokens")

    def __init__(self):
        self.ref = 0
        self.hash: Optional[int] = None
        self.tokens: List[int] = []


class Allocator:
    def __init__(self, num_blocks: int, block_size: int = 16):
        self.block_size = block_size
        self.blocks = [_Block() for _ in range(num_blocks)]
        # ref == 0 blocks, least recently released first; initially in id order
        self.pool: "OrderedDict[int, None]" = OrderedDict((i, None) for i in range(num_blocks))
        self.by_hash: dict = {}

    # ---- one physical block out of the pool (the LRU end)
    def _take(self) -> int:
        if not self.pool:
            raise MemoryError("no free KV cache block")
        bid, _ = self.pool.popitem(last=False)
        blk = self.blocks[bid]
        if blk.hash is not None:
            del self.by_hash[blk.hash]
            blk.hash = None
        blk.tokens = []
        blk.ref = 1
        return bid

    def allocate_for_prompt(self, token_ids) -> Tuple[List[int], int]:
        bs = self.block_size
        chunks = [[int(t) for t in token_ids[s:s + bs]] for s in range(0, len(token_ids), bs)]
        # count the hits and the hit blocks that sit in the pool, changing nothing
        n_hit, hits_in_pool, parent = 0, 0, 0
        for chunk in chunks:
            if len(chunk) < bs:
                break
            hit = self.by_hash.get(block_hash(parent, chunk))
            if hit is None:
                break
            n_hit += 1
            hits_in_pool += self.blocks[hit].ref == 0
            parent = self.blocks[hit].hash
        if len(chunks) - n_hit > len(self.pool) - hits_in_pool:
            raise MemoryError("no free KV cache block")

        table: List[int] = []
        cached = 0
        parent = 0
        matching = True
        for chunk in chunks:
            full = len(chunk) == bs
            if full and matching:
                h = block_hash(parent, chunk)
                hit = self.by_hash.get(h)
                if hit is not None:
                    if self.blocks[hit].ref == 0:
                        del self.pool[hit]
                    self.blocks[hit].ref += 1
                    table.append(hit)
                    cached += bs
                    parent = h
                    continue
                matching = False
            bid = self._take()
            blk = self.blocks[bid]
            blk.tokens = list(chunk)
            if full:
                h = block_hash(parent, chunk)
                blk.hash = h
                self.by_hash[h] = bid
                parent = h
            table.append(bid)
        return table, cached

    def append_slot(self, table: List[int], token: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        bs = self.block_size
        if not table or len(self.blocks[table[-1]].tokens) == bs:
            bid = self._take()
            self.blocks[bid].tokens.append(int(token))
            table.append(bid)
            return bid * bs, None
        last = table[-1]
        lb = self.blocks[last]
        if lb.ref > 1:
            bid = self._take()
            lb.ref -= 1
            nb = self.blocks[bid]
            nb.tokens = list(lb.tokens) + [int(token)]
            table[-1] = bid
            return bid * bs + len(nb.tokens) - 1, (last, bid)
        lb.tokens.append(int(token))
        return last * bs + len(lb.tokens) - 1, None

    def fork(self, table: List[int]) -> List[int]:
        for bid in table:
            self.blocks[bid].ref += 1
        return list(table)

    def free_sequence(self, table: List[int]) -> None:
        for bid in table:
            blk = self.blocks[bid]
            if blk.ref <= 0:
                raise ValueError(f"block {bid} is not held")
            blk.ref -= 1
            if blk.ref == 0:
                self.pool[bid] = None

    # ---- introspection
    def ref_count(self, bid: int) -> int:
        return self.blocks[bid].ref

    def hash_of(self, bid: int) -> Optional[int]:
        return self.blocks[bid].hash

    def num_tokens(self, bid: int) -> int:
        return len(self.blocks[bid].tokens)

    def free_order(self) -> List[int]:
        return list(self.pool.keys())

    def num_free(self) -> int:
        return len(self.pool)


def block_copy(k_cache: np.ndarray, v_cache: np.ndarray, pairs,
               k_scale: Optional[np.ndarray] = None, v_scale: Optional[np.ndarray] = None):
    """Copy every (src, dst) block of the pool, all heads and all 16 slots, in
    place: the device half of copy-on-write. Arrays are indexed by block
    first. Destinations are distinct and no destination is a source."""
    for src, dst in pairs:
        k_cache[dst] = k_cache[src]
        v_cache[dst] = v_cache[src]
        if k_scale is not None:
            k_scale[dst] = k_scale[src]
            v_scale[dst] = v_scale[src]
