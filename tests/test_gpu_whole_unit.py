"""The whole-unit grid: when no more (sequence, kv head) units than CTAs are
launched (and at least 3/4 as many) and the units are equally long within
3%, each CTA attends one unit whole. These cases size the batch from the
default grid of the device so that the rule applies, and compare the result
with the oracle, with a tolerance of 1e-2 (1 + |ref|) per element, and with
the cost-weighted split forced by an explicit CTA count."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import assert_close, gpu_pool
from workloads import Geometry, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _decode(w, pool, num_ctas=0):
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode(w.q().to(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                       torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, num_ctas=num_ctas, window=w.window)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return out.float().cpu().numpy()


@pytest.mark.parametrize("kv_dtype,n_kv,g,d_h,ragged,window", [
    ("bf16", 8, 8, 128, 0, 0),     # the Llama-3-70B layer shape
    ("bf16", 8, 4, 128, 5, 0),     # lengths differ by up to 5 tokens (one block)
    ("bf16", 4, 2, 64, 0, 600),    # windowed, equal windows
    ("int8", 8, 4, 128, 0, 0),
    ("int4", 8, 1, 128, 3, 0),
])
def test_whole_unit_grid_matches_oracle_and_split(kv_dtype, n_kv, g, d_h, ragged, window):
    geom = Geometry(n_h=n_kv * g, n_kv=n_kv, d_h=d_h, kv_dtype=kv_dtype)
    kc, _, _, _ = pa.allocate_pool(8, n_kv, d_h, kv_dtype, DEV)
    grid = pa.pa_decode_default_ctas(kc, geom.n_h, 8)
    B = max(1, (grid * 7 // 8) // n_kv)       # units = 7/8 of the grid
    assert 3 * grid <= 4 * B * n_kv <= 4 * grid
    rng = np.random.default_rng(B * 131 + n_kv)
    ctx = 1024 + rng.integers(0, ragged + 1, size=B)
    w = make_workload("whole_unit", geom, ctx, seed=7000 + B, window=window)
    pool = gpu_pool(w, DEV, fill_nan=True)
    got = _decode(w, pool)
    ref, st = oracle.decode_window(oracle.bf16_bits(w.q()), oracle.pool_for(w, fill_nan=True),
                                   w.block_tables, w.context_lens, geom.n_h, w.scale,
                                   window=window)
    assert st == 0
    assert_close(got, ref, f"whole-unit {kv_dtype} B{B}")
    split = _decode(w, pool, num_ctas=grid)
    assert_close(split, ref, f"split {kv_dtype} B{B}")
