"""Pins for the multi-query oracle (oracle_decode_mq): n_q new tokens per
sequence attend causally, as in speculative verification ("LLM 推理引擎设计",
§6) or a chunked-prefill chunk ("LLM 推理底层", "Chunked Prefill").
Query i of a sequence of ctx tokens attends positions 0 .. ctx - n_q + i."""
import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import Geometry, make_workload, random_queries


def qbits(B, n_q, n_h, d, seed=3):
    return oracle.bf16_bits(random_queries(seed, B * n_q, n_h, d)).reshape(B, n_q, n_h, d)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "int4"])
def test_each_query_is_a_single_query_decode_of_a_shorter_context(kv_dtype):
    w = make_workload("mq", Geometry(n_h=8, n_kv=2, d_h=64, kv_dtype=kv_dtype), [40, 17, 5, 64],
                      seed=2)
    pool = oracle.pool_for(w)
    n_q = 4
    q = qbits(w.B, n_q, 8, 64)
    out, st = oracle.decode_mq(q, pool, w.block_tables, w.context_lens, 8, w.scale)
    assert st == 0
    for i in range(n_q):
        ctx_i = np.maximum(w.context_lens - n_q + i + 1, 0).astype(np.int32)
        ref, st = oracle.decode(q[:, i], pool, w.block_tables, ctx_i, 8, w.scale)
        assert st == 0
        np.testing.assert_array_equal(out[:, i], ref)


def test_one_query_is_plain_decode():
    w = make_workload("mq", Geometry(n_h=4, n_kv=2, d_h=64), [5, 37], seed=4)
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    ref, _ = oracle.decode(q, pool, w.block_tables, w.context_lens, 4, w.scale)
    out, st = oracle.decode_mq(q[:, None], pool, w.block_tables, w.context_lens, 4, w.scale)
    assert st == 0 and np.array_equal(out[:, 0], ref)


def test_causal_mask_against_brute_force():
    w = make_workload("mq", Geometry(n_h=2, n_kv=1, d_h=64), [20, 3], seed=6)
    pool = oracle.pool_for(w)
    n_q = 5
    q = qbits(w.B, n_q, 2, 64, seed=9)
    out, st = oracle.decode_mq(q, pool, w.block_tables, w.context_lens, 2, w.scale)
    assert st == 0
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        k, v = w.seq_kv(b)
        kf = (oracle.bf16_bits(k).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        vf = (oracle.bf16_bits(v).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        for i in range(n_q):
            n = ctx - n_q + i + 1
            for h in range(2):
                qf = (q[b, i, h].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
                ref = brute.attend_rows(qf.tolist(), [kf[j, 0].tolist() for j in range(max(n, 0))],
                                        [vf[j, 0].tolist() for j in range(max(n, 0))], w.scale)
                np.testing.assert_allclose(out[b, i, h], ref, rtol=0, atol=1e-12)
                if n <= 0:  # ctx 3 < n_q 5: queries 0 and 1 see nothing
                    assert not out[b, i, h].any()
