"""pa_decode_noalloc: decode attention for callers that cannot allocate.

Some callers may not allocate device memory where they run decode attention
(a plugin whose host framework owns all device memory, a serving loop that
cannot afford an allocation mid-step). pa_decode_noalloc serves them with the
library's own fixed scratch array instead of a caller workspace. These tests
call it through the C ABI and check, on two calls in a row, that it returns
what pa_decode returns and what the CPU oracle computes, both within the
parity tolerance, and that a batch too big for the fixed array is refused
before any work is queued.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import TOL, assert_close, gpu_pool, oracle_full
from workloads import Geometry, make_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_cache_94_gb300 import build
    build.build()
    return torch.device("cuda:0")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _inputs(w, dev):
    pool = gpu_pool(w, dev)
    q = w.q("cpu").to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    return pool, q, bt, cl


def _noalloc(w, pool, q, bt, cl, dev):
    kc, vc, ks, vs = pool
    out = torch.full_like(q, float("nan"))
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    st = pa.library().pa_decode_noalloc(
        _p(q), _p(kc), _p(vc), _p(ks), _p(vs), _p(bt), bt.shape[1], _p(cl), w.B,
        ctypes.c_float(w.scale), _p(out), pa.geometry(kc, w.geom.n_h), _p(status), stream)
    assert st == 0, pa.library().pa_status_string(st)
    torch.cuda.synchronize(dev)
    assert int(status.item()) == 0
    return out


def _with_workspace(w, pool, q, bt, cl):
    kc, vc, ks, vs = pool
    out = pa.pa_decode(q, kc, vc, bt, cl, w.scale, k_scale=ks, v_scale=vs)
    torch.cuda.synchronize()
    return out


def test_noalloc_matches_pa_decode_two_calls_in_a_row(dev):
    # the second call has more (sequence, kv head) pairs than the first, so it
    # reuses scratch the first call left partial results in
    first = make_workload("noalloc_a", Geometry(32, 8, 128), [700, 3000, 41], seed=31)
    second = make_workload("noalloc_b", Geometry(32, 8, 128, kv_dtype="int8"),
                           [1, 900, 4000, 16, 2500, 333, 1200, 65, 3100, 2048], seed=32)
    for w in (first, second):
        pool, q, bt, cl = _inputs(w, dev)
        want = _with_workspace(w, pool, q, bt, cl).float()
        got = _noalloc(w, pool, q, bt, cl, dev).float()
        assert torch.isfinite(got).all()
        excess = (got - want).abs() - TOL * (1 + want.abs())
        assert excess.max().item() <= 0, f"{w.name}: max |d| {(got - want).abs().max().item()}"
        ref, _ = oracle_full(w)
        assert_close(got.cpu().numpy(), ref, f"{w.name} against the oracle")


def test_noalloc_refuses_batches_beyond_its_scratch(dev):
    g = pa.pa_geom(num_blocks=1024, n_h=128, n_kv=8, d_h=128, block_size=16, kv_dtype=0,
                   reserved=0)
    lib = pa.library()
    assert lib.pa_decode_workspace_size(g, 8192, 0) > (8 << 20)
    fake = ctypes.c_void_p(1 << 20)  # refused before any pointer is used
    st = lib.pa_decode_noalloc(fake, fake, fake, None, None, fake, 16, fake, 8192,
                               ctypes.c_float(0.1), fake, g, None, None)
    assert st == -7  # PA_ERR_WORKSPACE
