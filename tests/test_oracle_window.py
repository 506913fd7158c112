"""Pins for the sliding-window / attention-sink oracle (oracle_decode_window).

Sliding window: "kv-cache-guide" (guijiagi.com) §5.1, only the latest w
tokens are kept and attended. Attention sink: same page §4.3, the first k
tokens of an INT8 cache stay unquantised. Each pin checks the oracle against
something other than itself: a re-laid-out pool, the pure-Python brute
force, closed forms, and the plain oracle_decode where the two must agree.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import Geometry, make_workload, random_rows

BS = 16


def wl(kv_dtype, ctx, seed=3, n_h=4, n_kv=2, d_h=64):
    return make_workload("pin", Geometry(n_h=n_h, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype), ctx,
                         seed)


def rows_f(bits):
    """uint16 bf16 bits [..., d] -> float64."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def pool_row(pool, blk, kv, off):
    if pool.kv_dtype == "int8":
        return (pool.k[blk, kv, off].astype(np.float32) * pool.k_scale[blk, kv, off]).astype(np.float64), \
               (pool.v[blk, kv, off].astype(np.float32) * pool.v_scale[blk, kv, off]).astype(np.float64)
    return rows_f(pool.k[blk, kv, off]), rows_f(pool.v[blk, kv, off])


def sink_rows(w, n_sink, seed=77):
    """bf16 sink rows [B, n_kv, n_sink, d_h] (bits): any rows will do for the pins."""
    k, v = random_rows(seed, w.B * n_sink, w.geom.n_kv, w.geom.d_h)
    shp = (w.B, n_sink, w.geom.n_kv, w.geom.d_h)
    kb = oracle.bf16_bits(k).reshape(shp).transpose(0, 2, 1, 3)
    vb = oracle.bf16_bits(v).reshape(shp).transpose(0, 2, 1, 3)
    return np.ascontiguousarray(kb), np.ascontiguousarray(vb)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8"])
def test_no_window_equals_plain_decode(kv_dtype):
    w = wl(kv_dtype, [5, 37, 16, 1])
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    ref, st = oracle.decode(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    for window in (0, 37, 1000):
        out, st2 = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h,
                                        w.scale, window=window)
        assert st == st2 == 0
        assert np.array_equal(out, ref)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8"])
@pytest.mark.parametrize("window", [1, 7, 16, 20, 33])
def test_window_equals_decode_of_the_last_tokens(kv_dtype, window):
    # the window's tokens written into a fresh pool at positions 0..n-1
    w = wl(kv_dtype, [5, 37, 50])
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    out, st = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                   window=window)
    assert st == 0
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        start = max(0, ctx - window)
        k, v = w.seq_kv(b)
        n = ctx - start
        nblk = -(-n // BS)
        small = oracle.Pool(nblk, w.geom.n_kv, w.geom.d_h, BS, kv_dtype)
        assert small.write(oracle.bf16_bits(k[start:ctx]), oracle.bf16_bits(v[start:ctx]),
                           np.arange(n)) == 0
        ref, st = oracle.decode(q[b:b + 1], small, np.arange(nblk, dtype=np.int32)[None],
                                np.array([n], np.int32), w.geom.n_h, w.scale)
        assert st == 0
        np.testing.assert_allclose(out[b], ref[0], rtol=0, atol=1e-12)


def test_window_against_brute_force_and_closed_form():
    w = wl("bf16", [37, 9])
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    g = w.geom.n_h // w.geom.n_kv
    for window in (3, 1):
        out, st = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h,
                                       w.scale, window=window)
        assert st == 0
        for b in range(w.B):
            ctx = int(w.context_lens[b])
            k, v = w.seq_kv(b)
            kf, vf = rows_f(oracle.bf16_bits(k)), rows_f(oracle.bf16_bits(v))
            for h in range(w.geom.n_h):
                kv = h // g
                sel = range(max(0, ctx - window), ctx)
                ref = brute.attend_rows(rows_f(q[b, h]).tolist(), [kf[j, kv].tolist() for j in sel],
                                        [vf[j, kv].tolist() for j in sel], w.scale)
                np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)
                if window == 1:  # a single attended token: its V row, exactly
                    assert np.array_equal(out[b, h], vf[ctx - 1, kv])


def test_entries_before_the_window_are_never_read():
    w = wl("int8", [40, 70])
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    ref, _ = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                  window=20)
    bt = w.block_tables.copy()
    bt[0, :1] = -1          # window of sequence 0 starts at 20: block 0 unused
    bt[1, :3] = 10 ** 6     # window of sequence 1 starts at 50: blocks 0..2 unused
    out, st = oracle.decode_window(q, pool, bt, w.context_lens, w.geom.n_h, w.scale, window=20)
    assert st == 0 and np.array_equal(out, ref)
    bt[1, 3] = -1           # block 3 holds positions 48..63, inside the window
    out, st = oracle.decode_window(q, pool, bt, w.context_lens, w.geom.n_h, w.scale, window=20)
    assert st == 1 and not out[1].any() and np.array_equal(out[0], ref[0])


@pytest.mark.parametrize("n_sink,window", [(4, 0), (4, 6), (16, 0), (3, 40)])
def test_sink_rows_against_brute_force(n_sink, window):
    w = wl("int8", [2, 4, 21, 40])
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    sk, sv = sink_rows(w, n_sink)
    out, st = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                   window=window, n_sink=n_sink, sink_k_bits=sk, sink_v_bits=sv)
    assert st == 0
    g = w.geom.n_h // w.geom.n_kv
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        start = max(0, ctx - window) if window else 0
        for h in range(w.geom.n_h):
            kv = h // g
            ks, vs = [], []
            for j in range(start, ctx):
                if j < n_sink:
                    ks.append(rows_f(sk[b, kv, j]).tolist())
                    vs.append(rows_f(sv[b, kv, j]).tolist())
                else:
                    kr, vr = pool_row(pool, w.block_tables[b, j // BS], kv, j % BS)
                    ks.append(kr.tolist())
                    vs.append(vr.tolist())
            ref = brute.attend_rows(rows_f(q[b, h]).tolist(), ks, vs, w.scale)
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)


def test_sink_outside_the_window_changes_nothing():
    w = wl("int8", [40, 70])
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    sk, sv = sink_rows(w, 4)
    ref, _ = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                  window=30)
    out, st = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                   window=30, n_sink=4, sink_k_bits=sk, sink_v_bits=sv)
    assert st == 0 and np.array_equal(out, ref)
    # inside the window the sink rows do change the result
    out2, _ = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                   n_sink=4, sink_k_bits=sk, sink_v_bits=sv)
    full, _ = oracle.decode(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert not np.allclose(out2, full)
