"""GPU parity: the CUDA library through its C ABI against the CPU oracle.

Bit-exact: pool contents after pa_cache_write (bf16 rows, INT8 codes and
scales). Within |d| <= 1e-2 (1 + |ref|) per element: pa_decode outputs.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import (assert_close, gpu_decode, gpu_pool, oracle_full,
                               oracle_one_sequence, pool_bits)
from workloads import Geometry, make_workload, named_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_94_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _check_pool_bitexact(w, pool, opool):
    kc, vc, ks, vs = pool
    np.testing.assert_array_equal(pool_bits(kc), opool.k)
    np.testing.assert_array_equal(pool_bits(vc), opool.v)
    if w.geom.kv_dtype in ("int8", "int4"):
        np.testing.assert_array_equal(ks.cpu().numpy().view(np.uint32), opool.k_scale.view(np.uint32))
        np.testing.assert_array_equal(vs.cpu().numpy().view(np.uint32), opool.v_scale.view(np.uint32))


# ------------------------------------------------------------------ small cases
SMALL = [
    # (n_h, n_kv, d_h, dtype, context lengths)
    (4, 2, 64, "bf16", [5, 37]),
    (32, 8, 128, "bf16", [1, 15, 16, 17, 100, 257, 1000]),
    (64, 8, 128, "bf16", [2048, 33, 700]),
    (8, 8, 128, "bf16", [1, 300, 48]),
    (16, 8, 64, "bf16", [19, 260]),
    (32, 2, 128, "bf16", [5, 130, 999]),
    (32, 8, 128, "int8", [1, 17, 500, 1300]),
    (32, 32, 128, "int8", [16, 33, 777]),
    (8, 4, 64, "int8", [3, 64, 129]),
    (16, 1, 128, "int8", [40, 200]),
    (32, 8, 128, "int4", [1, 17, 500, 1300]),
    (32, 32, 128, "int4", [16, 33, 777]),
    (8, 4, 64, "int4", [3, 64, 129]),
    (16, 1, 128, "int4", [40, 200]),
    (8, 8, 64, "int4", [1, 31, 250]),
    (32, 2, 64, "int4", [7, 90]),
    (8, 4, 128, "bf16", [0, 40, 0, 16]),
]


@pytest.mark.parametrize("n_h,n_kv,d_h,dt,ctx", SMALL)
def test_small_parity(dev, n_h, n_kv, d_h, dt, ctx):
    w = make_workload("small", Geometry(n_h, n_kv, d_h, kv_dtype=dt), ctx,
                      seed=1000 + n_h * 7 + d_h + len(ctx))
    pool = gpu_pool(w, dev)
    ref, opool = oracle_full(w)
    _check_pool_bitexact(w, pool, opool)
    out, st = gpu_decode(w, pool, dev)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref, f"{n_h}/{n_kv}/{d_h}/{dt}")
    for b, c in enumerate(ctx):
        if c == 0:
            assert (out[b] == 0).all()


def test_tiny_config(dev):
    w = named_workload("tiny")
    pool = gpu_pool(w, dev)
    ref, opool = oracle_full(w)
    _check_pool_bitexact(w, pool, opool)
    out, st = gpu_decode(w, pool, dev)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref, "tiny")


@pytest.mark.parametrize("dt", ["bf16", "int8", "int4"])
def test_split_count_invariance(dev, dt):
    w = make_workload("split", Geometry(32, 8, 128, kv_dtype=dt), [3000, 17, 1500, 4096], seed=77)
    pool = gpu_pool(w, dev)
    ref, _ = oracle_full(w)
    outs = []
    for n in [1, 2, 3, 7, 64, 300, 1000, 0]:
        out, st = gpu_decode(w, pool, dev, num_ctas=n)
        assert st == 0
        assert_close(out.float().cpu().numpy(), ref, f"num_ctas={n}")
        outs.append(out.float())
    # one CTA per (sequence, kv head) would need no merge; all splits agree
    for o in outs[1:]:
        assert (o - outs[0]).abs().max().item() < 2e-2


def test_block_permutation_is_bit_identical(dev):
    w = make_workload("perm", Geometry(32, 8, 128), [900, 33, 1600], seed=5)
    pool = gpu_pool(w, dev)
    out1, _ = gpu_decode(w, pool, dev)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.num_blocks)
    kc, vc, ks, vs = pool
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    idx = torch.from_numpy(perm).to(dev)
    kc2[idx] = kc
    vc2[idx] = vc
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    out2, st = gpu_decode(w, (kc2, vc2, ks, vs), dev, table=bt)
    assert st == 0
    assert torch.equal(out1.view(torch.int16), out2.view(torch.int16))


@pytest.mark.parametrize("dt", ["bf16", "int8", "int4"])
def test_poisoned_pool(dev, dt):
    # unused slots and unused blocks hold NaN: never read, never propagated
    w = make_workload("nan", Geometry(32, 8, 128, kv_dtype=dt), [5, 17, 31, 250], seed=9,
                      pool_factor=2.0)
    clean, _ = gpu_decode(w, gpu_pool(w, dev), dev)
    dirty, st = gpu_decode(w, gpu_pool(w, dev, fill_nan=True), dev)
    assert st == 0
    assert torch.isfinite(dirty.float()).all()
    assert torch.equal(clean.view(torch.int16), dirty.view(torch.int16))


def test_repeated_calls_reuse_workspace(dev):
    # the counters are reset by each call: the same answer, call after call
    w = make_workload("rep", Geometry(64, 8, 128), [5000, 3000], seed=3)
    pool = gpu_pool(w, dev)
    first, _ = gpu_decode(w, pool, dev)
    for _ in range(5):
        again, st = gpu_decode(w, pool, dev)
        assert st == 0
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


def test_device_errors_are_reported_not_faulted(dev):
    w = make_workload("err", Geometry(8, 2, 64), [40, 40], seed=4)
    pool = gpu_pool(w, dev)
    ref, _ = oracle_full(w)
    # a block id outside the pool
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_blocks + 5
    out, st = gpu_decode(w, pool, dev, table=bt)
    assert pa.pa_status_from_device(st) == -5
    assert_close(out[0].float().cpu().numpy(), ref[0], "unaffected sequence")
    # a context length the table cannot hold
    out, st = gpu_decode(w, pool, dev, ctx=np.array([40, 10_000], np.int32))
    assert pa.pa_status_from_device(st) == -9
    assert (out[1] == 0).all()
    # a slot outside the pool
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    k = torch.ones(2, 2, 64, dtype=torch.bfloat16, device=dev)
    slots = torch.tensor([-1, w.num_blocks * 16], dtype=torch.int64, device=dev)
    before = kc.clone()
    pa.pa_cache_write(k, k, slots, kc, vc, ks, vs, dev_status=status)
    torch.cuda.synchronize()
    assert pa.pa_status_from_device(int(status.item())) == -6
    assert torch.equal(before.view(torch.int16), kc.view(torch.int16))


# ------------------------------------------------------------ full-size configs
@pytest.mark.parametrize("name", ["llama3_8b", "llama3_70b", "llama2_7b_int8_prefix",
                                  "long_context"])
def test_full_size_config_sampled(dev, name):
    w = named_workload(name)
    pool = gpu_pool(w, dev, gen_device=dev)
    out, st = gpu_decode(w, pool, dev, gen_device=dev)
    assert st == 0
    out = out.float().cpu().numpy()
    assert np.isfinite(out).all()
    rng = np.random.default_rng(0)
    picks = sorted(set([0, w.B - 1] + rng.choice(w.B, size=min(2, w.B), replace=False).tolist()))
    kc, vc, ks, vs = pool
    for b in picks:
        ref, opool = oracle_one_sequence(w, b, gen_device=dev)
        assert_close(out[b], ref, f"{name} seq {b}")
        # the sequence's tiles in the device pool equal the oracle's
        nblk = w.num_seq_blocks(b)
        phys = torch.from_numpy(w.block_tables[b, :nblk].astype(np.int64)).to(dev)
        np.testing.assert_array_equal(pool_bits(kc.index_select(0, phys)), opool.k)
        np.testing.assert_array_equal(pool_bits(vc.index_select(0, phys)), opool.v)
        if ks is not None:
            np.testing.assert_array_equal(ks.index_select(0, phys).cpu().numpy(), opool.k_scale)
            np.testing.assert_array_equal(vs.index_select(0, phys).cpu().numpy(), opool.v_scale)


@pytest.mark.parametrize("dt", ["bf16", "int8", "int4"])
def test_maximum_batch(dev, dt):
    # 8192 sequences (the largest batch the ABI takes), tiny and ragged
    # contexts, a few empty: the per-sequence prefix arrays are at their largest
    rng = np.random.default_rng(5)
    ctx = rng.integers(1, 40, 8192)
    ctx[[0, 1000, 8191]] = 0
    w = make_workload("maxb", Geometry(8, 2, 64, kv_dtype=dt), ctx.tolist(), seed=13)
    ref, _ = oracle_full(w)
    out, st = gpu_decode(w, gpu_pool(w, dev), dev)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref, f"{dt} B=8192")


def test_prepared_calls_repeat_on_new_contents(dev):
    # a Prepared call re-issues the same marshalled call: new input contents,
    # new result, identical to the direct call's
    w = make_workload("prep", Geometry(32, 8, 128), [300, 17, 1000], seed=19)
    kc, vc, ks, vs = gpu_pool(w, dev)
    q = w.q(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    out = torch.empty_like(q)
    call = pa.pa_decode(q, kc, vc, bt, cl, w.scale, out=out, prepare=True)
    assert isinstance(call, pa.Prepared)
    for seed in (1, 2):
        q.copy_(torch.randn(q.shape, generator=torch.Generator().manual_seed(seed)).to(q))
        got = call().clone()
        ref = pa.pa_decode(q, kc, vc, bt, cl, w.scale)
        torch.cuda.synchronize()
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
