"""GPU parity of sliding-window decode and INT8 attention-sink rows
(pa_decode_opt, pa_sink_write) against oracle_decode_window.

Sliding window: "kv-cache-guide" (guijiagi.com) §5.1; attention sink: same
page §4.3. Inputs are the seeded workloads; the sink rows are each
sequence's own first bf16 K/V rows, written on the device by pa_sink_write.
"""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import assert_close, gpu_pool
from workloads import Geometry, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def sink_inputs(w, n_sink):
    """Rows of positions < n_sink of every sequence: (k, v [T, n_kv, d], seq_rows, positions)."""
    ks, vs, rows, pos = [], [], [], []
    for b in range(w.B):
        n = min(n_sink, int(w.context_lens[b]))
        if n == 0:
            continue
        k, v = w.seq_kv(b)
        ks.append(k[:n])
        vs.append(v[:n])
        rows += [b] * n
        pos += list(range(n))
    return (torch.cat(ks), torch.cat(vs), np.array(rows, np.int32), np.array(pos, np.int32))


def oracle_sink_bits(w, n_sink, k, v, rows, pos):
    shp = (w.B, w.geom.n_kv, n_sink, w.geom.d_h)
    sk = np.zeros(shp, np.uint16)
    sv = np.zeros(shp, np.uint16)
    kb, vb = oracle.bf16_bits(k), oracle.bf16_bits(v)
    for t in range(len(rows)):
        sk[rows[t], :, pos[t]] = kb[t]
        sv[rows[t], :, pos[t]] = vb[t]
    return sk, sv


def run(w, pool, window=0, sink=None, num_ctas=0, table=None):
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    bt = w.block_tables if table is None else table
    out = pa.pa_decode(w.q().to(DEV), kc, vc, torch.from_numpy(bt).to(DEV),
                       torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, num_ctas=num_ctas, window=window,
                       sink_k=None if sink is None else sink[0],
                       sink_v=None if sink is None else sink[1])
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(status.item())


def poison_before_window(w, pool, window):
    """NaN into the device pool at the positions of each window's first block
    that lie before the window: the kernel must mask them, not just skip them."""
    kc, vc, ks, vs = pool
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        start = max(0, ctx - window)
        for j in range(start - start % 16, start):
            blk, off = int(w.block_tables[b, j // 16]), j % 16
            if kc.dtype == torch.bfloat16:
                kc[blk, :, off] = float("nan")
                vc[blk, :, off] = float("nan")
            else:
                ks[blk, :, off] = float("nan")
                vs[blk, :, off] = float("nan")


GEOMS = [("bf16", 128, 4), ("bf16", 64, 2), ("int8", 128, 1), ("int8", 64, 8), ("int4", 128, 4),
         ("int4", 64, 1)]


@pytest.mark.parametrize("kv_dtype,d_h,g", GEOMS)
@pytest.mark.parametrize("window", [1, 5, 16, 40, 100])
def test_window_matches_oracle(kv_dtype, d_h, g, window):
    n_kv = 2
    w = make_workload("win", Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype),
                      [1, 16, 17, 40, 63, 129, 300, 0], seed=17)
    pool = gpu_pool(w, DEV, fill_nan=True)
    opool = oracle.pool_for(w, fill_nan=True)
    poison_before_window(w, pool, window)
    ref, st = oracle.decode_window(oracle.bf16_bits(w.q()), opool, w.block_tables, w.context_lens,
                                   w.geom.n_h, w.scale, window=window)
    assert st == 0
    for num_ctas in (0, 1, 3, 50):
        out, dst = run(w, pool, window=window, num_ctas=num_ctas)
        assert dst == 0
        assert_close(out, ref, f"{kv_dtype} d{d_h} g{g} window {window} ctas {num_ctas}")


def test_window_never_reads_entries_before_it():
    w = make_workload("win", Geometry(n_h=8, n_kv=2, d_h=128), [300, 129, 40], seed=19)
    pool = gpu_pool(w, DEV)
    base, _ = run(w, pool, window=33)
    bt = w.block_tables.copy()
    for b in range(w.B):
        first = max(0, int(w.context_lens[b]) - 33) // 16
        bt[b, :first] = -7  # outside the pool: must not be read
    out, st = run(w, pool, window=33, table=bt)
    assert st == 0 and np.array_equal(out, base)


@pytest.mark.parametrize("kv_dtype,d_h,g", [("int8", 128, 1), ("int8", 128, 4), ("int8", 64, 8),
                                            ("int4", 128, 8), ("int4", 64, 2)])
@pytest.mark.parametrize("n_sink,window", [(4, 0), (4, 3), (16, 0), (4, 50), (1, 0)])
def test_sink_rows_match_oracle(kv_dtype, d_h, g, n_sink, window):
    n_kv = 2
    w = make_workload("sink", Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype),
                      [1, 2, 4, 5, 16, 21, 40, 200], seed=23)
    pool = gpu_pool(w, DEV, fill_nan=True)
    opool = oracle.pool_for(w, fill_nan=True)
    # the pool's own rows at sink positions must not be read: poison their scales
    for b in range(w.B):
        for j in range(min(n_sink, int(w.context_lens[b]))):
            blk = int(w.block_tables[b, j // 16])
            pool[2][blk, :, j % 16] = float("nan")
            pool[3][blk, :, j % 16] = float("nan")
    k, v, rows, pos = sink_inputs(w, n_sink)
    sk = torch.full((w.B, n_kv, n_sink, d_h), float("nan"), dtype=torch.bfloat16, device=DEV)
    sv = torch.full_like(sk, float("nan"))
    pa.pa_sink_write(k.to(DEV), v.to(DEV), torch.from_numpy(rows).to(DEV),
                     torch.from_numpy(pos).to(DEV), sk, sv)
    osk, osv = oracle_sink_bits(w, n_sink, k, v, rows, pos)
    torch.cuda.synchronize()
    # the written rows are the inputs, bit for bit
    got = sk.view(torch.int16).cpu().numpy().view(np.uint16)
    for t in range(len(rows)):
        assert np.array_equal(got[rows[t], :, pos[t]], osk[rows[t], :, pos[t]])
    ref, st = oracle.decode_window(oracle.bf16_bits(w.q()), opool, w.block_tables,
                                   w.context_lens, w.geom.n_h, w.scale, window=window,
                                   n_sink=n_sink, sink_k_bits=osk, sink_v_bits=osv)
    assert st == 0
    for num_ctas in (0, 1, 7, 64):
        out, dst = run(w, pool, window=window, sink=(sk, sv), num_ctas=num_ctas)
        assert dst == 0
        assert_close(out, ref, f"{kv_dtype} sink {n_sink} window {window} d{d_h} g{g} "
                               f"ctas {num_ctas}")


def test_decode_opt_argument_errors():
    w = make_workload("e", Geometry(n_h=4, n_kv=2, d_h=64), [20], seed=1)
    pool = gpu_pool(w, DEV)
    sk = torch.zeros((1, 2, 4, 64), dtype=torch.bfloat16, device=DEV)
    with pytest.raises(pa.PAError) as e:
        run(w, pool, sink=(sk, sk))  # sink rows on a bf16 pool
    assert e.value.status == -2
    with pytest.raises(pa.PAError) as e:
        run(w, pool, window=-1)
    assert e.value.status == -2


def test_long_context_window_sampled():
    # the pages' example: window 4096 over long contexts
    w = make_workload("lw", Geometry(n_h=32, n_kv=8, d_h=128), [32768, 20000, 4096, 100], seed=29)
    pool = gpu_pool(w, DEV)
    out, st = run(w, pool, window=4096)
    assert st == 0
    opool = oracle.pool_for(w)
    ref, st = oracle.decode_window(oracle.bf16_bits(w.q()), opool, w.block_tables,
                                   w.context_lens, w.geom.n_h, w.scale, window=4096)
    assert st == 0
    assert_close(out, ref, "long context window 4096")


def test_mistral_window_workload_sampled():
    # the bench workload, in the launch configuration the bench times
    from workloads import named_workload
    w = named_workload("mistral_7b_window")
    pool = gpu_pool(w, DEV, gen_device=DEV)
    out, st = run_named(w, pool)
    assert st == 0 and np.isfinite(out).all()
    g = w.geom
    for b in (0, 5, w.B - 1):
        k, v = w.seq_kv(b, DEV)
        ctx = int(w.context_lens[b])
        nblk = -(-ctx // 16)
        small = oracle.Pool(nblk, g.n_kv, g.d_h, 16, g.kv_dtype)
        assert small.write(oracle.bf16_bits(k), oracle.bf16_bits(v), np.arange(ctx)) == 0
        ref, st = oracle.decode_window(oracle.bf16_bits(w.q(DEV)[b:b + 1]), small,
                                       np.arange(nblk, dtype=np.int32)[None],
                                       np.array([ctx], np.int32), g.n_h, w.scale, window=w.window)
        assert st == 0
        assert_close(out[b], ref[0], f"mistral window seq {b}")


def run_named(w, pool):
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode(w.q(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                       torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, window=w.window)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(status.item())
