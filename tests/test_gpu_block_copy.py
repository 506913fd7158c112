"""GPU parity of the copy-on-write path: pa_block_copy against the oracle's
block copy, and a whole decode step driven by the native block manager
(prefix caching, fork, copy-on-write, cache write, decode) against the
oracle allocator, oracle pool and oracle decode on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
import workloads
from oracle.allocator import Allocator, block_copy as oracle_block_copy
from tests.gpu_helpers import assert_close, pool_bits

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
BS = 16


def random_pool(seed, nb, n_kv, d_h, kv_dtype):
    """Arbitrary pool contents (inputs only): numpy arrays k, v, k_scale, v_scale."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    shape = (nb, n_kv, BS, d_h)
    if kv_dtype == "bf16":
        k = torch.randn(shape, generator=gen).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        v = torch.randn(shape, generator=gen).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        return k, v, None, None
    if kv_dtype == "int4":  # two codes per byte
        shape = shape[:3] + (d_h // 2,)
        k = torch.randint(0, 256, shape, generator=gen, dtype=torch.uint8).numpy()
        v = torch.randint(0, 256, shape, generator=gen, dtype=torch.uint8).numpy()
    else:
        k = torch.randint(-128, 128, shape, generator=gen, dtype=torch.int8).numpy()
        v = torch.randint(-128, 128, shape, generator=gen, dtype=torch.int8).numpy()
    ks = torch.rand(shape[:3], generator=gen).numpy().astype(np.float32)
    vs = torch.rand(shape[:3], generator=gen).numpy().astype(np.float32)
    return k, v, ks, vs


def to_device(k, v, ks, vs):
    if k.dtype == np.uint16:
        kd = torch.from_numpy(k.view(np.int16)).view(torch.bfloat16).to(DEV)
        vd = torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(DEV)
        return kd, vd, None, None
    return (torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV),
            torch.from_numpy(ks).to(DEV), torch.from_numpy(vs).to(DEV))


@pytest.mark.parametrize("kv_dtype,n_kv,d_h,nb,npairs", [
    ("bf16", 8, 128, 1000, 300),   # Llama-3-8B layer: 32 KiB per block and tensor, two chunks
    ("bf16", 2, 64, 40, 7),
    ("int8", 32, 128, 300, 100),   # LLaMA-2-7B MHA layer: 64 KiB codes + 2 KiB scales
    ("int8", 1, 64, 16, 3),        # one 1 KiB tile, a partial chunk
    ("int4", 8, 128, 200, 50),     # 8 KiB of packed codes per block and tensor
    ("int4", 1, 64, 16, 3),        # one 512-byte tile
])
def test_block_copy_bit_exact(kv_dtype, n_kv, d_h, nb, npairs):
    k, v, ks, vs = random_pool(11, nb, n_kv, d_h, kv_dtype)
    pairs = workloads.block_copy_pairs(5, nb, npairs)
    kd, vd, ksd, vsd = to_device(k, v, ks, vs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_block_copy(kd, vd, torch.from_numpy(pairs).to(DEV), ksd, vsd, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    oracle_block_copy(k, v, pairs.tolist(), ks, vs)
    assert np.array_equal(pool_bits(kd), k) and np.array_equal(pool_bits(vd), v)
    if kv_dtype != "bf16":
        assert np.array_equal(ksd.cpu().numpy().view(np.uint32), ks.view(np.uint32))
        assert np.array_equal(vsd.cpu().numpy().view(np.uint32), vs.view(np.uint32))


def test_block_copy_skips_and_reports_bad_pairs():
    nb = 20
    k, v, ks, vs = random_pool(12, nb, 4, 128, "int8")
    pairs = np.array([[1, 2], [nb + 3, 4], [5, -1], [6, 7]], np.int32)
    kd, vd, ksd, vsd = to_device(k, v, ks, vs)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    pa.pa_block_copy(kd, vd, torch.from_numpy(pairs).to(DEV), ksd, vsd, dev_status=status)
    torch.cuda.synchronize()
    assert pa.pa_status_from_device(int(status.item())) == -5
    oracle_block_copy(k, v, [(1, 2), (6, 7)], ks, vs)  # the valid pairs only
    assert np.array_equal(pool_bits(kd), k) and np.array_equal(pool_bits(vd), v)
    assert np.array_equal(ksd.cpu().numpy(), ks) and np.array_equal(vsd.cpu().numpy(), vs)


def test_block_copy_empty_is_a_no_op():
    kd = torch.zeros((4, 2, BS, 64), dtype=torch.bfloat16, device=DEV)
    vd = torch.zeros_like(kd)
    pa.pa_block_copy(kd, vd, torch.zeros((0, 2), dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert not kd.any()


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "int4"])
def test_decode_step_with_prefix_cache_fork_and_copy_on_write(kv_dtype):
    n_h, n_kv, d_h, NB, CAP = 8, 2, 128, 64, 12
    vocab = np.random.default_rng(21)
    system = vocab.integers(0, 1000, 2 * BS + 5).tolist()     # 2 full blocks + 5 tokens
    other = system[:2 * BS] + vocab.integers(0, 1000, 9).tolist()

    nat, ora = pa.BlockAllocator(NB), Allocator(NB)
    kc, vc, ksc, vsc = pa.allocate_pool(NB, n_kv, d_h, kv_dtype, DEV)
    opool = oracle.Pool(NB, n_kv, d_h, BS, kv_dtype)

    def write_both(rows_seed, table_n, table_o, first, n_tok):
        # rows for positions first..n_tok-1 at the slots each side's table gives
        if n_tok <= first:
            return
        k, v = workloads.random_rows(rows_seed, n_tok - first, n_kv, d_h)
        pos = np.arange(first, n_tok)
        sn = np.asarray(table_n)[pos // BS].astype(np.int64) * BS + pos % BS
        so = np.asarray(table_o)[pos // BS].astype(np.int64) * BS + pos % BS
        assert np.array_equal(sn, so)
        pa.pa_cache_write(k.to(DEV), v.to(DEV), torch.from_numpy(sn).to(DEV), kc, vc, ksc, vsc)
        assert opool.write(oracle.bf16_bits(k), oracle.bf16_bits(v), so) == 0

    # prefill of two prompts: the second hits the first's two full blocks
    tn0, c0 = nat.allocate_prompt(system)
    to0, _ = ora.allocate_for_prompt(system)
    write_both(100, tn0, to0, c0, len(system))
    tn1, c1 = nat.allocate_prompt(other)
    to1, oc1 = ora.allocate_for_prompt(other)
    assert c1 == oc1 == 2 * BS and tn1.tolist() == to1
    write_both(101, tn1, to1, c1, len(other))
    # parallel sampling: three more branches of the first prompt
    tabs_n = [tn0] + [nat.fork(tn0) for _ in range(3)] + [tn1]
    tabs_o = [to0] + [ora.fork(to0) for _ in range(3)] + [to1]
    ntok = [len(system)] * 4 + [len(other)]

    # one decode step: append, copy-on-write, write the new rows, attend
    B = len(tabs_n)
    tables = np.full((B, CAP), 0, np.int32)
    nblk = np.array([len(t) for t in tabs_n], np.int32)
    for i, t in enumerate(tabs_n):
        tables[i, :len(t)] = t
    new_tok = [7, 8, 9, 10, 11]
    slots, cow = nat.append_slots(tables, nblk, new_tok)
    exp_slots, exp_cow = [], []
    for i, t in enumerate(tabs_o):
        s, c = ora.append_slot(t, new_tok[i])
        exp_slots.append(s)
        if c is not None:
            exp_cow.append(c)
    assert slots.tolist() == exp_slots and [tuple(x) for x in cow.tolist()] == exp_cow
    assert len(exp_cow) == 3  # three of the four branches copy the shared tail

    pa.pa_block_copy(kc, vc, torch.from_numpy(cow).to(DEV), ksc, vsc)
    oracle_block_copy(opool.k, opool.v, exp_cow, opool.k_scale, opool.v_scale)
    k_new, v_new = workloads.random_rows(102, B, n_kv, d_h)
    pa.pa_cache_write(k_new.to(DEV), v_new.to(DEV), torch.from_numpy(slots).to(DEV), kc, vc, ksc, vsc)
    assert opool.write(oracle.bf16_bits(k_new), oracle.bf16_bits(v_new),
                       np.array(exp_slots, np.int64)) == 0
    ctx = np.array(ntok, np.int32) + 1

    q = workloads.random_queries(103, B, n_h, d_h)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode(q.to(DEV), kc, vc, torch.from_numpy(tables).to(DEV),
                       torch.from_numpy(ctx).to(DEV), d_h ** -0.5, k_scale=ksc, v_scale=vsc,
                       dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0

    otab = np.zeros((B, CAP), np.int32)
    for i, t in enumerate(tabs_o):
        otab[i, :len(t)] = t
    assert np.array_equal(otab, tables)
    ref, st = oracle.decode(oracle.bf16_bits(q), opool, otab, ctx, n_h, d_h ** -0.5)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref, f"{kv_dtype} CoW decode step")
    # the pools agree bit for bit on every block a table names
    used = sorted({int(b) for i in range(B) for b in tables[i, :nblk[i]]})
    assert np.array_equal(pool_bits(kc)[used], opool.k[used])
    assert np.array_equal(pool_bits(vc)[used], opool.v[used])
    if kv_dtype != "bf16":
        assert np.array_equal(ksc.cpu().numpy()[used], opool.k_scale[used])
    # the four branches now differ only in their last token
    assert len({int(tables[i, nblk[i] - 1]) for i in range(4)}) == 4
