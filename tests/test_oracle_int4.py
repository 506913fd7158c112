"""Pins for the INT4 oracle: quantiser, nibble packing and INT4 decode.

"kv-cache-guide" (guijiagi.com) §4.2 `quantize_kv_cache` with num_bits == 4:
scale = max|x| / 7 per (token, head) row, code = clamp(round(x / scale), -8, 7),
dequantised as code * scale. The pages say only that INT4 halves INT8's bytes;
the cache packs element 2i in the low nibble of byte i (two's complement).
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import Geometry, make_workload


def bits_of(values):
    return oracle.bf16_bits(torch.tensor(values, dtype=torch.float32).to(torch.bfloat16))


def test_int4_ties_round_half_to_even():
    # amax 7 -> scale exactly 1: x / scale = x, so ties are visible directly
    x = bits_of([7.0, 0.5, 1.5, 2.5, -2.5, -0.5, -3.5, 6.5])
    code, sc = oracle.quantize_row_int4(x)
    assert sc == np.float32(1.0)
    assert code.tolist() == [7, 0, 2, 2, -2, 0, -4, 6]


def test_int4_zero_row_and_amax_code():
    code, sc = oracle.quantize_row_int4(bits_of([0.0] * 8))
    assert sc == 0.0 and not code.any()
    rng = np.random.default_rng(1)
    for _ in range(50):
        x = bits_of(rng.standard_normal(64).tolist())
        code, sc = oracle.quantize_row_int4(x)
        xf = (x.astype(np.uint32) << 16).view(np.float32)
        i = int(np.argmax(np.abs(xf)))
        assert abs(int(code[i])) == 7 and np.sign(code[i]) == np.sign(xf[i])
        assert code.min() >= -7 and code.max() <= 7
        # round trip within half a step (plus fp32 rounding of the quotient)
        err = np.abs(xf.astype(np.float64) - code.astype(np.float64) * np.float64(sc))
        assert (err <= sc / 2 * (1 + 1e-6) + 1e-30).all()


def test_int4_packing_nibble_order():
    # one token, one head: codes [1, -1, 7, -7, 0, 3, -2, 4] at amax 7
    vals = [1.0, -1.0, 7.0, -7.0, 0.0, 3.0, -2.0, 4.0]
    pool = oracle.Pool(1, 1, 8, 16, "int4")
    x = bits_of(vals).reshape(1, 1, 8)
    assert pool.write(x, x, np.array([3], np.int64)) == 0
    assert pool.k[0, 0, 3].tolist() == [0xF1, 0x97, 0x30, 0x4E]
    assert pool.k_scale[0, 0, 3] == np.float32(1.0)
    assert not pool.k[0, 0, :3].any() and not pool.k[0, 0, 4:].any()


def test_int4_halves_int8_bytes():
    # M = 2 L n_kv d_h S B b: INT4 stores b = 1/2 byte per element (4x less than fp16)
    m16 = oracle.kv_bytes(32, 8, 128, 4096, 1, 2)
    assert oracle.kv_bytes(32, 8, 128, 4096, 1, 0.5) * 4 == m16


def dequant(pool, blk, kv, off):
    out = []
    for which, sc in ((pool.k, pool.k_scale), (pool.v, pool.v_scale)):
        b = which[blk, kv, off]
        nib = np.stack([b & 15, b >> 4], axis=1).reshape(-1).astype(np.int32)
        code = np.where(nib >= 8, nib - 16, nib)
        out.append((code.astype(np.float32) * sc[blk, kv, off]).astype(np.float64))
    return out


@pytest.mark.parametrize("g", [1, 4])
def test_int4_decode_against_brute_force(g):
    w = make_workload("i4", Geometry(n_h=2 * g, n_kv=2, d_h=64, kv_dtype="int4"), [1, 19, 40],
                      seed=5)
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    out, st = oracle.decode(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        for h in range(w.geom.n_h):
            kv = h // g
            rows = [dequant(pool, w.block_tables[b, j // 16], kv, j % 16) for j in range(ctx)]
            qf = (q[b, h].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            ref = brute.attend_rows(qf.tolist(), [r[0].tolist() for r in rows],
                                    [r[1].tolist() for r in rows], w.scale)
            np.testing.assert_allclose(out[b, h], ref, rtol=0, atol=1e-12)


def test_int4_error_against_bf16_is_bounded():
    # dequantised INT4 rows differ from the bf16 rows by at most scale/2 each,
    # so the INT4 output stays near the bf16 output (a loose sanity bound)
    w = make_workload("i4", Geometry(n_h=4, n_kv=2, d_h=64, kv_dtype="int4"), [64], seed=6)
    wb = make_workload("b", Geometry(n_h=4, n_kv=2, d_h=64), [64], seed=6)
    o4, _ = oracle.decode(oracle.bf16_bits(w.q()), oracle.pool_for(w), w.block_tables,
                          w.context_lens, 4, w.scale)
    ob, _ = oracle.decode(oracle.bf16_bits(wb.q()), oracle.pool_for(wb), wb.block_tables,
                          wb.context_lens, 4, wb.scale)
    assert np.abs(o4 - ob).max() < 0.5
