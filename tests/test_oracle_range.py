"""CPU checks of the oracle on the dynamic-range inputs the GPU parity tests
use (workloads.PROFILES), before any GPU compares against it:

  * the closed forms: q = 0 and identical keys give the mean of the attended
    V rows, the one-hot query at scale 50 gives the matching key's V row;
  * the "rising" staircase makes the running maximum of the scores climb by
    more than 8 log2 units at least three times per sequence and head;
  * the oracle's raw scores reproduce its decode output through a softmax
    written here with numpy ("LLM 推理底层", "自回归解码与 KV Cache 的物理来源",
    eq. for o_t), and equal a brute-force dot product on a tiny case;
  * the v_range and kv_range rows span at least four decades of per-token
    magnitude, and q_big / q_small move q by the stated factors.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests.range_cases import (POOLS, assert_rising, closed_form, dequant_rows, run_oracle,
                               workload)
from workloads import Geometry, make_workload


@pytest.mark.parametrize("mode", ["plain", "window", "mq", "share"])
@pytest.mark.parametrize("profile", ["q_zero", "same_keys", "onehot"])
@pytest.mark.parametrize("kv_dtype", POOLS)
def test_oracle_meets_closed_forms(mode, profile, kv_dtype):
    w = workload("cf", 11, kv_dtype, 64, 8 if mode != "mq" else 2, profile, mode)
    ref, _ = run_oracle(w, mode)
    cf = closed_form(w, mode)
    assert np.abs(ref - cf).max() <= 1e-9 * (1 + np.abs(cf).max())


@pytest.mark.parametrize("mode", ["plain", "window", "share"])
@pytest.mark.parametrize("kv_dtype", POOLS)
@pytest.mark.parametrize("d_h", [64, 128])
def test_rising_profile_climbs(mode, kv_dtype, d_h):
    w = workload("rise", 12, kv_dtype, d_h, 8, "rising", mode)
    _, pool = run_oracle(w, mode)
    assert_rising(w, pool)


def test_normal_profile_does_not_climb():
    # the plain N(0, 1) inputs never reach a re-base: that is why the
    # profiles exist
    w = make_workload("flat", Geometry(16, 2, 128), [700, 1201], seed=13)
    pool = oracle.pool_for(w)
    s, st = oracle.scores(oracle.bf16_bits(w.q()), pool, w.block_tables, w.context_lens, 16,
                          w.scale)
    assert st == 0
    spread = np.nanmax(s, axis=2) - np.nanmin(s, axis=2)
    assert spread.max() / math.log(2) < 16


@pytest.mark.parametrize("kv_dtype", POOLS)
def test_scores_reproduce_decode(kv_dtype):
    w = workload("sc", 14, kv_dtype, 64, 8, "rising", "plain")
    pool = oracle.pool_for(w)
    q = oracle.bf16_bits(w.q())
    s, st = oracle.scores(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    out, st = oracle.decode(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        assert np.isnan(s[b, :, ctx:]).all()
        _, v = w.seq_kv(b)
        vd = dequant_rows(v, kv_dtype)               # [ctx, n_kv, d]
        for h in range(w.geom.n_h):
            x = s[b, h, :ctx]
            p = np.exp(x - x.max())
            p /= p.sum()
            np.testing.assert_allclose(p @ vd[:, h // w.geom.g], out[b, h], rtol=1e-10,
                                       atol=1e-12)


def test_scores_brute_force_tiny():
    w = make_workload("tiny_sc", Geometry(4, 2, 8), [5, 19], seed=15, num_blocks=4)
    pool = oracle.pool_for(w)
    q = w.q()
    s, st = oracle.scores(oracle.bf16_bits(q), pool, w.block_tables, w.context_lens, 4, 0.3)
    assert st == 0
    for b in range(2):
        k, _ = w.seq_kv(b)
        for h in range(4):
            for j in range(int(w.context_lens[b])):
                dot = sum(float(q[b, h, d]) * float(k[j, h // 2, d]) for d in range(8))
                assert abs(s[b, h, j] - 0.3 * dot) <= 1e-12 * (1 + abs(dot))


def test_scores_flag_bad_blocks():
    w = make_workload("bad_sc", Geometry(2, 1, 16), [20, 20], seed=16)
    pool = oracle.pool_for(w)
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_blocks
    s, st = oracle.scores(oracle.bf16_bits(w.q()), pool, bt, w.context_lens, 2, w.scale)
    assert st == oracle.BAD_BLOCK
    assert np.isnan(s[1]).all() and np.isfinite(s[0]).all()


def test_range_profiles_span_decades():
    for prof in ("v_range", "kv_range"):
        w = make_workload("amp", Geometry(4, 2, 64), [2000], seed=17, profile=prof)
        k, v = w.seq_kv(0)
        vm = v.float().abs().amax(-1)
        assert vm.max() / vm.min() > 1e4
        km = k.float().abs().amax(-1)
        assert (km.max() / km.min() > 1e4) == (prof == "kv_range")
    base = make_workload("qb", Geometry(4, 2, 64), [10], seed=18).q().float()
    big = make_workload("qb", Geometry(4, 2, 64), [10], seed=18, profile="q_big").q().float()
    small = make_workload("qb", Geometry(4, 2, 64), [10], seed=18, profile="q_small").q().float()
    torch.testing.assert_close(big / 1e3, base, rtol=1e-2, atol=0)
    torch.testing.assert_close(small * 1e3, base, rtol=1e-2, atol=1e-6)


def test_sink_outlier_first_token_dominates():
    w = make_workload("sink", Geometry(8, 2, 128), [4096], seed=19, profile="sink_outlier")
    pool = oracle.pool_for(w)
    s, st = oracle.scores(oracle.bf16_bits(w.q()), pool, w.block_tables, w.context_lens, 8,
                          w.scale)
    assert st == 0
    x = s[0]
    assert (x[:, 0] > x[:, 1:].max(axis=1) + 5).all()
