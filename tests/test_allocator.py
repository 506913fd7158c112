"""The native block manager (include/pa_alloc.h) against the oracle allocator.

Host only: the allocator never touches the GPU. Both sides run the same
seeded sequences of operations; block tables, cached-token counts, slots,
copy-on-write pairs, reference counts, fill counts, hashes and the order of
the evictable pool must agree exactly after every step, and a failing call
must fail on both sides and change nothing.
"""
import random

import numpy as np
import pytest

import paged_kv_cache_94_gb300 as pa
from oracle.allocator import Allocator, block_hash
from paged_kv_cache_94_gb300 import build as pa_build

BS = 16


@pytest.fixture(scope="module", autouse=True)
def _built():
    pa_build.build()


def same_state(nat: pa.BlockAllocator, ora: Allocator):
    assert nat.free_order() == ora.free_order()
    assert nat.num_free() == ora.num_free()
    for b in range(len(ora.blocks)):
        assert nat.block_info(b) == (ora.ref_count(b), ora.num_tokens(b), ora.hash_of(b)), b


def test_chained_hash_matches_the_oracle():
    rng = random.Random(3)
    for n in [0, 1, 15, 16, 29, 30, 31, 32, 33, 64, 200]:
        toks = [rng.randrange(1 << 31) for _ in range(n)]
        parent = rng.randrange(1 << 64)
        assert pa.block_hash(parent, toks) == block_hash(parent, toks)
    assert pa.block_hash(0, list(range(16))) == block_hash(0, list(range(16)))


def test_prompt_sharing_and_copy_on_write_match():
    nat, ora = pa.BlockAllocator(64), Allocator(64)
    prompt = list(range(500))
    tn, cn = nat.allocate_prompt(prompt)
    to, co = ora.allocate_for_prompt(prompt)
    assert tn.tolist() == to and cn == co == 0
    branches_o = [to] + [ora.fork(to) for _ in range(3)]
    branches_n = [tn] + [nat.fork(tn) for _ in range(3)]
    cap = 40
    tables = np.full((4, cap), -1, np.int32)
    nb = np.array([len(t) for t in branches_n], np.int32)
    for i, t in enumerate(branches_n):
        tables[i, :len(t)] = t
    slots, cow = nat.append_slots(tables, nb, [900, 901, 902, 903])
    exp_slots, exp_cow = [], []
    for i, t in enumerate(branches_o):
        s, c = ora.append_slot(t, 900 + i)
        exp_slots.append(s)
        if c is not None:
            exp_cow.append(c)
    assert slots.tolist() == exp_slots
    assert [tuple(x) for x in cow.tolist()] == exp_cow and len(exp_cow) == 3
    for i, t in enumerate(branches_o):
        assert tables[i, :nb[i]].tolist() == t
    same_state(nat, ora)
    # a second prompt with the same first 496 tokens hits 31 cached blocks
    t2n, c2n = nat.allocate_prompt(prompt[:496] + [1, 2, 3])
    t2o, c2o = ora.allocate_for_prompt(prompt[:496] + [1, 2, 3])
    assert t2n.tolist() == t2o and c2n == c2o == 496
    same_state(nat, ora)


def test_failures_match_and_change_nothing():
    nat, ora = pa.BlockAllocator(6), Allocator(6)
    t, _ = nat.allocate_prompt(list(range(3 * BS)))
    ora.allocate_for_prompt(list(range(3 * BS)))
    with pytest.raises(pa.PAError) as e:
        nat.allocate_prompt(list(range(1000, 1000 + 4 * BS)))
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
    with pytest.raises(MemoryError):
        ora.allocate_for_prompt(list(range(1000, 1000 + 4 * BS)))
    same_state(nat, ora)
    # a block nobody holds, and one named more often than it is held
    with pytest.raises(pa.PAError) as e:
        nat.free([5])
    assert e.value.status == pa.PA_ERR_STATE
    with pytest.raises(pa.PAError) as e:
        nat.free([int(t[0]), int(t[0])])
    assert e.value.status == pa.PA_ERR_STATE
    with pytest.raises(pa.PAError) as e:
        nat.fork([99])
    assert e.value.status == pa.PA_ERR_STATE
    with pytest.raises(pa.PAError) as e:
        nat.allocate_prompt([1, -2, 3])
    assert e.value.status == -2
    same_state(nat, ora)
    # a batch that runs out part-way keeps the sequences it finished
    tables = np.full((4, 8), -1, np.int32)
    nb = np.zeros(4, np.int32)
    with pytest.raises(pa.PAError) as e:
        nat.append_slots(tables, nb, [1, 2, 3, 4])
    assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS and e.value.num_done == 3
    assert nb.tolist() == [1, 1, 1, 0]
    # a full table with no room for a new block
    tables = np.array([t], np.int32)
    with pytest.raises(pa.PAError) as e:
        nat.append_slots(tables, np.array([3], np.int32), [7])
    assert e.value.status == -2 and e.value.num_done == 0


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_random_operation_sequences_match(seed):
    rng = random.Random(seed)
    NB, CAP = 80, 24
    nat, ora = pa.BlockAllocator(NB), Allocator(NB)
    prompts = [[rng.randrange(40) for _ in range(rng.randrange(0, 8 * BS))] for _ in range(5)]
    live_o, live_n = [], []  # oracle tables (lists); native rows (array, count)
    for step in range(400):
        op = rng.random()
        if op < 0.2 or not live_o:
            p = rng.choice(prompts) + [rng.randrange(40) for _ in range(rng.randrange(3))]
            try:
                to, co = ora.allocate_for_prompt(p)
            except MemoryError:
                with pytest.raises(pa.PAError) as e:
                    nat.allocate_prompt(p)
                assert e.value.status == pa.PA_ERR_OUT_OF_BLOCKS
            else:
                tn, cn = nat.allocate_prompt(p)
                assert tn.tolist() == to and cn == co
                live_o.append(to)
                row = np.full(CAP, -1, np.int32)
                row[:len(tn)] = tn
                live_n.append([row, len(tn)])
        elif op < 0.3:
            i = rng.randrange(len(live_o))
            live_o.append(ora.fork(live_o[i]))
            tn = nat.fork(live_n[i][0][:live_n[i][1]])
            row = np.full(CAP, -1, np.int32)
            row[:len(tn)] = tn
            live_n.append([row, len(tn)])
        elif op < 0.8:
            idx = rng.sample(range(len(live_o)), rng.randrange(1, min(4, len(live_o)) + 1))
            idx = [i for i in idx if len(live_o[i]) < CAP]
            if not idx:
                continue
            toks = [rng.randrange(40) for _ in idx]
            tables = np.stack([live_n[i][0] for i in idx])
            nb = np.array([live_n[i][1] for i in idx], np.int32)
            exp_slots, exp_cow, done = [], [], len(idx)
            for k, i in enumerate(idx):
                try:
                    s, c = ora.append_slot(live_o[i], toks[k])
                except MemoryError:
                    done = k
                    break
                exp_slots.append(s)
                if c is not None:
                    exp_cow.append(c)
            if done < len(idx):
                with pytest.raises(pa.PAError) as e:
                    nat.append_slots(tables, nb, toks)
                assert e.value.num_done == done
                assert [tuple(x) for x in e.value.cow_pairs.tolist()] == exp_cow
            else:
                slots, cow = nat.append_slots(tables, nb, toks)
                assert slots.tolist() == exp_slots
                assert [tuple(x) for x in cow.tolist()] == exp_cow
            for k, i in enumerate(idx):
                live_n[i] = [tables[k].copy(), int(nb[k])]
                assert live_n[i][0][:live_n[i][1]].tolist() == live_o[i]
        else:
            i = rng.randrange(len(live_o))
            ora.free_sequence(live_o.pop(i))
            row, n = live_n.pop(i)
            nat.free(row[:n])
        same_state(nat, ora)
