"""Seeded random parity sweep: pool type, head dim, group size, kv heads,
batch, a mix of context lengths around block edges, forced CTA counts and
sliding windows, each decode against the oracle on the same inputs."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import assert_close, gpu_pool
from workloads import Geometry, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
EDGES = [0, 1, 2, 15, 16, 17, 31, 32, 33, 255, 256, 257]


def draw(seed):
    rng = np.random.default_rng(1000 + seed)
    kv_dtype = ["bf16", "int8", "int4"][seed % 3]
    d_h = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    n_kv = int(rng.choice([1, 2, 4]))
    B = int(rng.integers(1, 20))
    ctx = [int(rng.choice(EDGES)) if rng.random() < 0.5 else int(rng.integers(1, 3000))
           for _ in range(B)]
    num_ctas = int(rng.choice([0, 1, 7, 300]))
    window = int(rng.choice([0, 0, 16, 100, 1024]))
    return kv_dtype, d_h, g, n_kv, ctx, num_ctas, window


@pytest.mark.parametrize("seed", range(48))
def test_random_decode_matches_oracle(seed):
    kv_dtype, d_h, g, n_kv, ctx, num_ctas, window = draw(seed)
    w = make_workload(f"fuzz{seed}", Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype),
                      ctx, seed=500 + seed, window=window)
    kc, vc, ks, vs = gpu_pool(w, DEV, fill_nan=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode(w.q().to(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                       torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, num_ctas=num_ctas, window=window)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, st = oracle.decode_window(oracle.bf16_bits(w.q()), oracle.pool_for(w, fill_nan=True),
                                   w.block_tables, w.context_lens, w.geom.n_h, w.scale,
                                   window=window)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref,
                 f"{kv_dtype} d{d_h} g{g} n_kv{n_kv} ctas{num_ctas} window{window} ctx{ctx}")


def draw_groups(rng, B):
    """Runs of adjacent sequences sharing a prefix of whole blocks (group id
    per sequence, -1: none): one block short of, at, or beyond the 8-block
    minimum, so some runs form groups and some do not."""
    groups, prefix, g_id, b = [], [], 0, 0
    while b < B:
        n = int(rng.integers(1, 6))
        shared = 16 * int(rng.choice([0, 6, 7, 8, 9, 19, 63]))
        for _ in range(min(n, B - b)):
            groups.append(g_id if (n > 1 and shared > 0) else -1)
            prefix.append(shared if (n > 1 and shared > 0) else 0)
            b += 1
        g_id += 1
    return groups, prefix


@pytest.mark.parametrize("seed", range(24))
def test_random_shared_prefix_matches_oracle(seed):
    rng = np.random.default_rng(2000 + seed)
    kv_dtype = ["bf16", "int8", "int4"][seed % 3]
    d_h = int(rng.choice([64, 128]))
    g = int(rng.choice([1, 2, 4, 8]))
    n_kv = int(rng.choice([1, 2]))
    B = int(rng.integers(2, 24))
    groups, prefix = draw_groups(rng, B)
    suffix = [int(rng.choice([1, 2, 16, 17])) if rng.random() < 0.4 else int(rng.integers(1, 400))
              for _ in range(B)]
    ctx = [p + s for p, s in zip(prefix, suffix)]
    w = make_workload(f"fshare{seed}", Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype),
                      ctx, seed=700 + seed, prefix_len=prefix, group=groups)
    kc, vc, ks, vs = gpu_pool(w, DEV, fill_nan=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode(w.q().to(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                       torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, share_prefix=True,
                       num_ctas=int(rng.choice([0, 1, 9, 250])))
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, st = oracle.decode(oracle.bf16_bits(w.q()), oracle.pool_for(w, fill_nan=True),
                            w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref, f"{kv_dtype} d{d_h} g{g} groups{groups} ctx{ctx}")


@pytest.mark.parametrize("seed", range(18))
def test_random_multi_query_matches_oracle(seed):
    rng = np.random.default_rng(3000 + seed)
    kv_dtype = ["bf16", "int8", "int4"][seed % 3]
    d_h = int(rng.choice([64, 128]))
    g, n_q = [(1, 2), (1, 4), (1, 8), (2, 2), (2, 4), (2, 8), (4, 2), (4, 4), (8, 2)][
        int(rng.integers(0, 9))]
    n_kv = int(rng.choice([1, 2]))
    B = int(rng.integers(1, 12))
    ctx = [int(rng.choice(EDGES)) if rng.random() < 0.5 else int(rng.integers(1, 2000))
           for _ in range(B)]
    w = make_workload(f"fmq{seed}", Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype),
                      ctx, seed=900 + seed, n_q=n_q)
    kc, vc, ks, vs = gpu_pool(w, DEV, fill_nan=True)
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode_mq(w.q().to(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                          torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks,
                          v_scale=vs, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref, st = oracle.decode_mq(oracle.bf16_bits(w.q()), oracle.pool_for(w, fill_nan=True),
                               w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    assert_close(out.float().cpu().numpy(), ref, f"{kv_dtype} d{d_h} g{g} n_q{n_q} ctx{ctx}")
