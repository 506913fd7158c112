"""Pins for the oracle block allocator (oracle/allocator.py).

Each test checks a behaviour the pages state for prefix caching, copy-on-write
and block sharing ("LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention
调度", section "Prefix Caching 与 Copy-on-Write"; the vLLM interview page,
考点 4 on beam search), or an invariant that any correct allocator keeps.
"""
import random
import struct

import numpy as np
import pytest

from oracle.allocator import Allocator, block_copy, block_hash, hash_input

BS = 16


def chain(tokens):
    """H_0, H_1, ... over the full blocks of `tokens`."""
    out, parent = [], 0
    for s in range(0, len(tokens) - len(tokens) % BS, BS):
        parent = block_hash(parent, tokens[s:s + BS])
        out.append(parent)
    return out


def snapshot(a: Allocator):
    return ([(b.ref, b.hash, list(b.tokens)) for b in a.blocks], a.free_order(), dict(a.by_hash))


def check_invariants(a: Allocator, tables):
    refs = np.zeros(len(a.blocks), np.int64)
    for t in tables:
        for bid in t:
            refs[bid] += 1
    assert [b.ref for b in a.blocks] == refs.tolist()
    assert sorted(a.free_order()) == [i for i in range(len(a.blocks)) if refs[i] == 0]
    for h, bid in a.by_hash.items():
        assert a.blocks[bid].hash == h
        assert len(a.blocks[bid].tokens) == BS
    assert sum(1 for b in a.blocks if b.hash is not None) == len(a.by_hash)


def test_hash_byte_layout():
    # parent 7 as 8 little-endian bytes, then the ids 1 and 258 (0x102) as
    # 4 little-endian bytes each, written out by hand
    assert hash_input(7, [1, 258]).hex() == "0700000000000000" "01000000" "02010000"
    assert hash_input(0, []).hex() == "0000000000000000"
    assert hash_input(2**64 - 1, [2**31 - 1]).hex() == "ffffffffffffffff" "ffffff7f"
    # the digest is an 8-byte BLAKE2b of exactly those bytes, read little-endian:
    # it changes with every byte and never depends on anything else
    base = block_hash(7, [1, 258])
    assert 0 <= base < 2**64
    assert block_hash(7, [1, 258]) == base
    assert len({base, block_hash(7, [1, 259]), block_hash(6, [1, 258]),
                block_hash(7, [258, 1]), block_hash(7, [1, 258, 0])}) == 5


def test_hash_chain_identifies_prefixes():
    rng = random.Random(1)
    a = [rng.randrange(32000) for _ in range(8 * BS)]
    assert chain(a) == chain(list(a))
    # one changed token in block 3 changes H_3 and every later H, not the earlier ones
    b = list(a)
    b[3 * BS + 5] ^= 1
    ca, cb = chain(a), chain(b)
    assert ca[:3] == cb[:3]
    assert all(x != y for x, y in zip(ca[3:], cb[3:]))
    # equal block contents under different parents hash differently
    c = a[BS:2 * BS] + a[BS:2 * BS]
    hc = chain(c)
    assert hc[0] != hc[1]
    # swapping two blocks changes the chain from the first swapped block on
    d = a[BS:2 * BS] + a[:BS] + a[2 * BS:]
    assert chain(d)[0] != ca[0] and chain(d)[1] != ca[1]


def test_beam_search_shares_prefix():
    # beam = 4 over a 512-token common prefix (32 blocks): the four branches
    # hold the same 32 physical blocks, four references each, instead of 128 blocks
    a = Allocator(200)
    prompt = list(range(512))
    t0, cached = a.allocate_for_prompt(prompt)
    assert cached == 0 and len(t0) == 32
    branches = [t0] + [a.fork(t0) for _ in range(3)]
    assert a.num_free() == 200 - 32
    assert all(a.ref_count(b) == 4 for b in t0)
    # the prefix ends on a block boundary: each branch's next token opens a new block, no copy
    for i, t in enumerate(branches):
        slot, cow = a.append_slot(t, 7 + i)
        assert cow is None and slot % BS == 0 and len(t) == 33
    assert a.num_free() == 200 - 36
    check_invariants(a, branches)


def test_copy_on_write_of_shared_partial_tail():
    a = Allocator(100)
    t0, _ = a.allocate_for_prompt(list(range(500)))  # 31 full blocks + 4 tokens
    assert len(t0) == 32 and a.num_tokens(t0[-1]) == 4
    tail = t0[-1]
    branches = [t0] + [a.fork(t0) for _ in range(3)]
    cows = []
    for i, t in enumerate(branches):
        slot, cow = a.append_slot(t, 900 + i)
        assert slot % BS == 4  # the new token takes offset 500 mod 16 of its own tail
        cows.append(cow)
    # the first three writers copy the shared tail; the last holder writes in place
    assert all(c is not None and c[0] == tail for c in cows[:3])
    assert len({c[1] for c in cows[:3]}) == 3
    assert cows[3] is None and branches[3][-1] == tail
    assert a.ref_count(tail) == 1
    assert a.num_free() == 100 - 35
    for i, t in enumerate(branches):
        assert a.blocks[t[-1]].tokens == [496, 497, 498, 499, 900 + i]
        assert t[:31] == t0[:31]
    check_invariants(a, branches)


def test_prefix_cache_hits_until_first_miss():
    a = Allocator(64)
    sys_prompt = [5000 + i for i in range(4 * BS)]
    t1, c1 = a.allocate_for_prompt(sys_prompt + [1, 2, 3])
    t2, c2 = a.allocate_for_prompt(sys_prompt + [7, 8])
    assert c1 == 0 and c2 == 4 * BS
    assert t2[:4] == t1[:4] and t2[4] != t1[4]
    assert all(a.ref_count(b) == 2 for b in t1[:4])
    # a miss in block 1 ends matching: block 2 is not reused even though its
    # tokens are the same (its chained hash differs anyway)
    p3 = list(sys_prompt)
    p3[BS] += 1
    t3, c3 = a.allocate_for_prompt(p3)
    assert c3 == BS and t3[0] == t1[0] and t3[1] != t1[1] and t3[2] != t1[2]
    # only full blocks are matched: a partial tail never hits
    t4, c4 = a.allocate_for_prompt(sys_prompt + [1, 2, 3])
    assert c4 == 4 * BS and t4[4] != t1[4]
    check_invariants(a, [t1, t2, t3, t4])


def test_released_blocks_stay_cached_until_evicted():
    a = Allocator(11)
    p = list(range(3 * BS))
    t1, _ = a.allocate_for_prompt(p)
    a.free_sequence(t1)
    assert a.free_order()[-3:] == t1  # released in table order, at the recent end
    t2, c2 = a.allocate_for_prompt(p)
    assert c2 == 3 * BS and t2 == t1  # reused from the evictable pool
    a.free_sequence(t2)
    # taking every other free block first evicts the oldest released ones
    other, _ = a.allocate_for_prompt(list(range(100000, 100000 + 9 * BS)))
    assert t1[0] in other and t1[1] not in other and t1[2] not in other
    assert a.hash_of(t1[0]) is not None and a.hash_of(t1[0]) != chain(p)[0]
    assert a.hash_of(t1[1]) == chain(p)[1]  # still cached, but unreachable without H_0
    a.free_sequence(other)
    t3, c3 = a.allocate_for_prompt(p)
    assert c3 == 0  # H_0 was evicted with block t1[0], so matching stops at once
    assert t3 == [t1[1], t1[2], other[0]]
    check_invariants(a, [t3])


def test_out_of_blocks_leaves_state_unchanged():
    a = Allocator(6)
    t1, _ = a.allocate_for_prompt(list(range(3 * BS)))
    before = snapshot(a)
    with pytest.raises(MemoryError):
        a.allocate_for_prompt(list(range(10000, 10000 + 4 * BS)))
    assert snapshot(a) == before
    # three hits plus three new blocks fit exactly in the three free blocks
    t2, c2 = a.allocate_for_prompt(list(range(3 * BS)) + list(range(7, 7 + 2 * BS + 1)))
    assert c2 == 3 * BS and t2[:3] == t1 and a.num_free() == 0
    a.free_sequence(t2)
    # a hit block that sits in the pool cannot also be taken as a new block
    a.free_sequence(t1)
    before = snapshot(a)
    with pytest.raises(MemoryError):
        a.allocate_for_prompt(list(range(3 * BS)) + list(range(500, 500 + 3 * BS + 1)))
    assert snapshot(a) == before
    t1, c1 = a.allocate_for_prompt(list(range(3 * BS)) + list(range(500, 500 + 3 * BS)))
    assert c1 == 3 * BS and a.num_free() == 0
    t2 = a.fork(t1)
    a2 = Allocator(1)
    tt, _ = a2.allocate_for_prompt(list(range(BS)))
    s = snapshot(a2)
    with pytest.raises(MemoryError):
        a2.append_slot(tt, 3)
    assert snapshot(a2) == s
    check_invariants(a, [t1, t2])


def test_random_operations_keep_invariants():
    rng = random.Random(94)
    a = Allocator(96)
    live = []
    prompts = [[rng.randrange(50) for _ in range(rng.randrange(0, 6 * BS))] for _ in range(6)]
    for _ in range(600):
        op = rng.random()
        try:
            if op < 0.25 or not live:
                base = rng.choice(prompts)
                t, c = a.allocate_for_prompt(base + [rng.randrange(50) for _ in range(rng.randrange(3))])
                assert c % BS == 0 and c <= len(base) + 2
                live.append(t)
            elif op < 0.35:
                live.append(a.fork(rng.choice(live)))
            elif op < 0.8:
                t = rng.choice(live)
                n_before = len(t)
                slot, cow = a.append_slot(t, rng.randrange(50))
                assert slot // BS == t[-1] and len(t) in (n_before, n_before + 1)
                if cow is not None:
                    assert cow[1] == t[-1] and a.ref_count(cow[0]) >= 1
            else:
                a.free_sequence(live.pop(rng.randrange(len(live))))
        except MemoryError:
            a.free_sequence(live.pop(0))
        check_invariants(a, live)


def test_block_copy_oracle():
    rng = np.random.default_rng(0)
    k = rng.standard_normal((6, 2, BS, 8)).astype(np.float32)
    v = rng.standard_normal((6, 2, BS, 8)).astype(np.float32)
    k0, v0 = k.copy(), v.copy()
    block_copy(k, v, [(1, 4), (2, 5)])
    assert np.array_equal(k[4], k0[1]) and np.array_equal(v[5], v0[2])
    assert np.array_equal(k[:4], k0[:4]) and np.array_equal(v[:4], v0[:4])

