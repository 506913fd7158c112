"""GPU parity of multi-query decode (pa_decode_mq) against oracle_decode_mq:
n_q new tokens per sequence attending causally ("LLM 推理引擎设计" §6,
speculative verification; "LLM 推理底层" "Chunked Prefill")."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import assert_close, gpu_pool
from workloads import Geometry, make_workload, named_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(w, pool, table=None, gen_device="cpu"):
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    bt = w.block_tables if table is None else table
    # the same generator device as the oracle's inputs (CPU and CUDA streams differ)
    out = pa.pa_decode_mq(w.q(gen_device).to(DEV), kc, vc, torch.from_numpy(bt).to(DEV),
                          torch.from_numpy(w.context_lens).to(DEV), w.scale, dev_status=status,
                          k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(status.item())


MQ_CASES = [(1, 2, 128), (1, 8, 128), (2, 4, 64), (4, 4, 128), (8, 2, 128), (4, 2, 64),
            (2, 8, 128), (1, 4, 64)]


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "int4"])
@pytest.mark.parametrize("g,n_q,d_h", MQ_CASES)
def test_mq_matches_oracle(g, n_q, d_h, kv_dtype):
    n_kv = 2
    # contexts: shorter than n_q, one block, a block plus one, odd tails, long
    w = make_workload("mq", Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype),
                      [1, 3, 8, 16, 17, 33, 47, 100, 1000, 0], seed=31 + g + n_q, n_q=n_q)
    pool = gpu_pool(w, DEV, fill_nan=True)
    out, st = run(w, pool)
    assert st == 0
    ref, ost = oracle.decode_mq(oracle.bf16_bits(w.q()), oracle.pool_for(w, fill_nan=True),
                                w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert ost == 0
    assert_close(out, ref, f"{kv_dtype} g{g} n_q{n_q} d{d_h}")
    # tokens whose causal range is empty (ctx < n_q - i) and empty sequences give zeros
    for b, ctx in enumerate(w.context_lens):
        for i in range(n_q):
            if ctx - n_q + i + 1 <= 0:
                assert not out[b, i].any()


def test_mq_with_one_query_equals_decode():
    w = make_workload("mq1", Geometry(n_h=32, n_kv=8, d_h=128), [700, 33, 1600], seed=8)
    pool = gpu_pool(w, DEV)
    kc, vc, _, _ = pool
    q = w.q(DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cl = torch.from_numpy(w.context_lens).to(DEV)
    a = pa.pa_decode(q, kc, vc, bt, cl, w.scale)
    b = pa.pa_decode_mq(q[:, None], kc, vc, bt, cl, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b[:, 0].view(torch.int16))


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "int4"])
def test_mq_unsupported_shapes_are_refused(kv_dtype):
    # g * n_q = 32 query rows per kv head, and n_q = 3: not compiled
    for g, n_q in ((4, 8), (2, 3)):
        w = make_workload("mqx", Geometry(n_h=2 * g, n_kv=2, d_h=64, kv_dtype=kv_dtype), [20],
                          seed=3, n_q=n_q)
        kc, vc, ks, vs = gpu_pool(w, DEV)
        with pytest.raises(pa.PAError):
            pa.pa_decode_mq(w.q().to(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                            torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks,
                            v_scale=vs)


@pytest.mark.parametrize("kv_dtype", ["int8", "int4"])
def test_mq_quantised_with_one_query_equals_decode(kv_dtype):
    w = make_workload("mq1q", Geometry(n_h=32, n_kv=8, d_h=128, kv_dtype=kv_dtype),
                      [700, 33, 1600, 5], seed=9)
    kc, vc, ks, vs = gpu_pool(w, DEV)
    q = w.q(DEV)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cl = torch.from_numpy(w.context_lens).to(DEV)
    a = pa.pa_decode(q, kc, vc, bt, cl, w.scale, k_scale=ks, v_scale=vs)
    b = pa.pa_decode_mq(q[:, None], kc, vc, bt, cl, w.scale, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b[:, 0].view(torch.int16))


def test_speculative_verify_workload_sampled():
    w = named_workload("llama3_8b_spec4")
    pool = gpu_pool(w, DEV, gen_device=DEV)
    out, st = run(w, pool, gen_device=DEV)
    assert st == 0 and np.isfinite(out).all()
    g = w.geom
    for b in (0, 17, w.B - 1):
        k, v = w.seq_kv(b, DEV)
        ctx = int(w.context_lens[b])
        nblk = -(-ctx // 16)
        small = oracle.Pool(nblk, g.n_kv, g.d_h, 16, g.kv_dtype)
        assert small.write(oracle.bf16_bits(k), oracle.bf16_bits(v), np.arange(ctx)) == 0
        ref, st = oracle.decode_mq(oracle.bf16_bits(w.q(DEV)[b:b + 1]), small,
                                   np.arange(nblk, dtype=np.int32)[None], np.array([ctx], np.int32),
                                   g.n_h, w.scale)
        assert st == 0
        assert_close(out[b], ref[0], f"spec4 seq {b}")
