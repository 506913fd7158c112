"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests retypes the oracle's formula: each compares it with a
printed value from the pages, a closed form, a library routine, an invariant,
or the independent pure-Python brute force.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import brute
from workloads import Geometry, make_workload, named_workload

pytestmark = pytest.mark.filterwarnings("ignore::DeprecationWarning")


def _bits(t):
    return oracle.bf16_bits(t)


# --------------------------------------------------------------- byte formula
def test_kv_bytes_match_printed_values(golden_dir):
    data = json.load(open(os.path.join(golden_dir, "kv_bytes.json")))
    for c in data["cases"]:
        got = oracle.kv_bytes(c["L"], c["n_kv"], c["d_h"], c["S"], c["B"], c["b"])
        if "exact" in c:
            assert got == c["exact"], c["cite"]
        else:
            printed = c["printed"] * c["unit"]
            assert abs(got - printed) <= c["rel_tol"] * printed, c["cite"]
    for e in data["errata"]:
        got = oracle.kv_bytes(e["L"], e["n_kv"], e["d_h"], e["S"], e["B"], e["b"])
        assert got == e["formula_value"]
        assert abs(got - e["printed_wrong"]) > 1e9  # the printed figure is not the formula's


def test_kv_bytes_int4_half_byte():
    # kv-cache-guide §2.1 lists INT4 = 0.5 bytes per element
    assert oracle.kv_bytes(1, 8, 128, 2, 1, 0.5) == 2 * 8 * 128 * 2 * 0.5


# ------------------------------------------------------- write_kv worked example
def test_write_kv_worked_example(golden_dir):
    ex = json.load(open(os.path.join(golden_dir, "write_kv_example.json")))
    for table, expect_phys in ((ex["block_table"], ex["block_table"][1]),
                               (ex["variant_block_table"], ex["variant_expected_phys"])):
        pool = oracle.Pool(ex["num_blocks"], ex["n_heads"], ex["head_dim"], ex["block_size"])
        j = ex["token_idx"]
        bs = ex["block_size"]
        assert j // bs == ex["expected_logical_block"] and j % bs == ex["expected_offset"]
        # the block manager's slot for token j of this request
        slot = table[j // bs] * bs + j % bs
        k = torch.full((1, ex["n_heads"], ex["head_dim"]), ex["k_fill"]).bfloat16()
        v = torch.full((1, ex["n_heads"], ex["head_dim"]), ex["v_fill"]).bfloat16()
        assert pool.write(_bits(k), _bits(v), np.array([slot])) == 0
        kf = torch.from_numpy(pool.k.view(np.int16)).view(torch.bfloat16).float().numpy()
        vf = torch.from_numpy(pool.v.view(np.int16)).view(torch.bfloat16).float().numpy()
        assert kf[expect_phys, :, ex["expected_offset"], :].mean() == ex["expected_k_mean"]
        assert vf[expect_phys, :, ex["expected_offset"], :].mean() == ex["expected_v_mean"]
        # nothing else was written
        mask = np.ones(kf.shape, bool)
        mask[expect_phys, :, ex["expected_offset"], :] = False
        assert (kf[mask] == 0).all() and (vf[mask] == 0).all()


def test_write_skips_negative_and_flags_out_of_range_slots():
    pool = oracle.Pool(2, 1, 8, 16)
    k = torch.ones(3, 1, 8).bfloat16()
    st = pool.write(_bits(k), _bits(k), np.array([-1, 31, 32]))
    assert st == oracle.BAD_SLOT
    assert pool.k[1, 0, 15].view(np.int16).tolist() == _bits(k[0, 0]).view(np.int16).tolist()
    assert int(np.count_nonzero(pool.k)) == 8


# ----------------------------------------------------------------- INT8 quant
def test_int8_hand_ties(golden_dir):
    data = json.load(open(os.path.join(golden_dir, "int8_ties.json")))
    for r in data["rows"]:
        x = torch.tensor(r["x"], dtype=torch.float32).bfloat16()
        assert x.float().tolist() == [float(a) for a in r["x"]]  # exact in bf16
        code, sc = oracle.quantize_row_int8(_bits(x))
        assert float(sc) == r["scale"]
        assert code.tolist() == r["codes"]


def _torch_quant_rows(x_bf16):
    """The page's quantiser run by torch in fp32 (kv-cache-guide §4.2)."""
    xf = x_bf16.float()
    scale = xf.abs().max(dim=-1, keepdim=True).values / 127
    q = (xf / scale).round().clamp(-128, 127).to(torch.int8)
    return q, scale.squeeze(-1)


def test_int8_matches_torch_fp32_on_random_rows():
    g = torch.Generator().manual_seed(3)
    x = (torch.randn(512, 128, generator=g) * torch.logspace(-3, 3, 512).unsqueeze(1)).bfloat16()
    qt, st = _torch_quant_rows(x)
    for i in range(x.shape[0]):
        code, sc = oracle.quantize_row_int8(_bits(x[i]))
        assert np.float32(sc) == np.float32(st[i].item())
        assert (code == qt[i].numpy()).all(), i


def test_int8_roundtrip_bound_and_extremes():
    g = torch.Generator().manual_seed(4)
    x = torch.randn(64, 64, generator=g).bfloat16()
    for i in range(64):
        code, sc = oracle.quantize_row_int8(_bits(x[i]))
        xf = x[i].float().numpy()
        deq = code.astype(np.float32) * np.float32(sc)
        # rounding to the nearest integer code: error at most half a step, plus
        # the fp32 rounding of the product code*scale
        assert np.all(np.abs(xf - deq) <= 0.5 * sc + 2 * np.spacing(np.abs(xf)))
        j = int(np.argmax(np.abs(xf)))
        assert abs(int(code[j])) == 127
        assert code.min() >= -127


# ------------------------------------------------------------ decode attention
def _sdpa_reference(w, device="cpu", dequant_int8=False):
    """softmax(q K^T * scale) V per sequence on the CONTIGUOUS history, by torch's
    scaled_dot_product_attention in float64 (kv-cache-guide §1.2 KVCache.attention)."""
    g = w.geom
    q = w.q(device).double()
    outs = []
    for b in range(w.B):
        k, v = w.seq_kv(b, device)
        if dequant_int8:
            kq, ks = _torch_quant_rows(k)
            vq, vs = _torch_quant_rows(v)
            k = (kq.float() * ks.unsqueeze(-1)).double()
            v = (vq.float() * vs.unsqueeze(-1)).double()
        else:
            k, v = k.double(), v.double()
        ctx = k.shape[0]
        if ctx == 0:
            outs.append(torch.zeros(g.n_h, g.d_h, dtype=torch.float64))
            continue
        # [n_h, ctx, d] with kv head h // g for query head h
        kk = k.permute(1, 0, 2).repeat_interleave(g.g, dim=0)
        vv = v.permute(1, 0, 2).repeat_interleave(g.g, dim=0)
        o = torch.nn.functional.scaled_dot_product_attention(
            q[b].unsqueeze(1), kk, vv, scale=w.scale)
        outs.append(o.squeeze(1))
    return torch.stack(outs).numpy()


def _oracle_out(w, fill_nan=False, table=None):
    pool = oracle.pool_for(w, fill_nan=fill_nan)
    bt = w.block_tables if table is None else table
    out, st = oracle.decode(_bits(w.q()), pool, bt, w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    return out


@pytest.mark.parametrize("n_h,n_kv,d_h", [(4, 2, 64), (8, 1, 64), (4, 4, 32), (16, 2, 16)])
def test_paged_oracle_equals_contiguous_sdpa(n_h, n_kv, d_h):
    w = make_workload("t", Geometry(n_h, n_kv, d_h), [1, 15, 16, 17, 40], seed=11 + n_h)
    out = _oracle_out(w)
    ref = _sdpa_reference(w)
    np.testing.assert_allclose(out, ref, rtol=1e-10, atol=1e-12)


def test_tiny_config_equals_sdpa():
    w = named_workload("tiny")
    np.testing.assert_allclose(_oracle_out(w), _sdpa_reference(w), rtol=1e-10, atol=1e-12)


def test_int8_paged_oracle_equals_dequantised_sdpa():
    w = make_workload("t8", Geometry(4, 2, 64, kv_dtype="int8"), [3, 16, 33], seed=5)
    out = _oracle_out(w)
    ref = _sdpa_reference(w, dequant_int8=True)
    np.testing.assert_allclose(out, ref, rtol=1e-9, atol=1e-11)


def test_shared_prefix_workload_equals_sdpa():
    w = make_workload("pfx", Geometry(2, 2, 32, kv_dtype="int8"), [40, 50, 35, 36], seed=6,
                      prefix_len=[32, 32, 32, 32], group=[0, 0, 1, 1])
    # the two groups' prefix blocks are shared between their sequences
    assert (w.block_tables[0, :2] == w.block_tables[1, :2]).all()
    assert (w.block_tables[2, :2] == w.block_tables[3, :2]).all()
    np.testing.assert_allclose(_oracle_out(w), _sdpa_reference(w, dequant_int8=True),
                               rtol=1e-9, atol=1e-11)


def test_brute_force_matches_c_oracle():
    w = named_workload("tiny")
    pool = oracle.pool_for(w)
    out, st = oracle.decode(_bits(w.q()), pool, w.block_tables, w.context_lens, 4, w.scale)
    bf = brute.paged_decode(_bits(w.q()), pool.k, pool.v, w.block_tables, w.context_lens, 4, 2,
                            w.scale)
    np.testing.assert_allclose(out, np.array(bf), rtol=1e-12, atol=1e-14)


def test_permutation_of_physical_blocks_leaves_output_unchanged():
    w = make_workload("perm", Geometry(4, 2, 32), [7, 33, 48], seed=21)
    base = _oracle_out(w)
    # move every physical block to a new id: relabel the pool and the table
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    pool = oracle.pool_for(w)
    pool2 = oracle.Pool(w.num_blocks, 2, 32)
    pool2.k[perm] = pool.k
    pool2.v[perm] = pool.v
    bt = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    out2, st = oracle.decode(_bits(w.q()), pool2, bt, w.context_lens, 4, w.scale)
    assert st == 0
    np.testing.assert_array_equal(out2, base)


def test_unused_slots_and_blocks_never_read():
    w = make_workload("poison", Geometry(4, 2, 32), [5, 17, 31], seed=8, pool_factor=2.0)
    clean = _oracle_out(w)
    poisoned = _oracle_out(w, fill_nan=True)
    assert np.isfinite(poisoned).all()
    np.testing.assert_array_equal(poisoned, clean)


def _single_seq_pool(keys, vals, block_size=16):
    """A pool whose block table is 0,1,2,... for one sequence of given rows."""
    ctx, n_kv, d = keys.shape
    nb = -(-ctx // block_size)
    pool = oracle.Pool(nb, n_kv, d, block_size)
    pool.write(_bits(keys), _bits(vals), np.arange(ctx))
    return pool, np.arange(nb, dtype=np.int32)[None, :]


def test_closed_forms():
    g = torch.Generator().manual_seed(9)
    d = 32
    ctx = 37
    vals = torch.randn(ctx, 1, d, generator=g).bfloat16()
    vmean = vals.double().mean(0)[0].numpy()
    # identical keys -> uniform weights -> mean of V
    key = torch.randn(1, 1, d, generator=g).bfloat16().expand(ctx, 1, d).contiguous()
    pool, bt = _single_seq_pool(key, vals)
    q = torch.randn(1, 2, d, generator=g).bfloat16()
    out, _ = oracle.decode(_bits(q), pool, bt, np.array([ctx], np.int32), 2, 1 / math.sqrt(d))
    np.testing.assert_allclose(out[0, 0], vmean, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(out[0, 1], vmean, rtol=1e-12, atol=1e-13)
    # q = 0 -> mean of V whatever the keys
    keys = torch.randn(ctx, 1, d, generator=g).bfloat16()
    pool, bt = _single_seq_pool(keys, vals)
    out, _ = oracle.decode(_bits(torch.zeros(1, 1, d).bfloat16()), pool, bt,
                           np.array([ctx], np.int32), 1, 0.125)
    np.testing.assert_allclose(out[0, 0], vmean, rtol=1e-12, atol=1e-13)
    # ctx = 1 -> v_0
    out, _ = oracle.decode(_bits(q[:, :1]), pool, bt, np.array([1], np.int32), 1, 0.125)
    np.testing.assert_array_equal(out[0, 0], vals[0, 0].double().numpy())
    # ctx = 0 -> zeros
    out, _ = oracle.decode(_bits(q[:, :1]), pool, bt, np.array([0], np.int32), 1, 0.125)
    assert (out == 0).all()
    # a one-hot query matching one key, with a large scale -> that key's value
    keys = torch.zeros(ctx, 1, d)
    for j in range(ctx):
        keys[j, 0, j % d] = 1.0
    keys[20, 0, :] = 0
    keys[20, 0, 5] = 2.0
    pool, bt = _single_seq_pool(keys.bfloat16(), vals)
    qh = torch.zeros(1, 1, d)
    qh[0, 0, 5] = 1.0
    out, _ = oracle.decode(_bits(qh.bfloat16()), pool, bt, np.array([ctx], np.int32), 1, 50.0)
    np.testing.assert_allclose(out[0, 0], vals[20, 0].double().numpy(), atol=1e-15 + 1e-20)


def test_output_shifts_with_v():
    # the weights sum to one, so adding c to every V row adds c to the output
    g = torch.Generator().manual_seed(10)
    d, ctx = 16, 20
    keys = torch.randn(ctx, 1, d, generator=g).bfloat16()
    vals = torch.randint(-8, 8, (ctx, 1, d), generator=g).float()  # small ints: exact in bf16
    q = torch.randn(1, 1, d, generator=g).bfloat16()
    pool, bt = _single_seq_pool(keys, vals.bfloat16())
    o1, _ = oracle.decode(_bits(q), pool, bt, np.array([ctx], np.int32), 1, 0.25)
    pool2, _ = _single_seq_pool(keys, (vals + 4.0).bfloat16())
    o2, _ = oracle.decode(_bits(q), pool2, bt, np.array([ctx], np.int32), 1, 0.25)
    np.testing.assert_allclose(o2 - o1, 4.0, rtol=0, atol=1e-12)


def test_decode_flags_bad_blocks_and_contexts():
    w = make_workload("bad", Geometry(2, 1, 16), [20, 20], seed=2)
    pool = oracle.pool_for(w)
    bt = w.block_tables.copy()
    bt[1, 1] = w.num_blocks  # out of range
    out, st = oracle.decode(_bits(w.q()), pool, bt, w.context_lens, 2, w.scale)
    assert st == oracle.BAD_BLOCK
    assert (out[1] == 0).all() and np.abs(out[0]).sum() > 0
    out, st = oracle.decode(_bits(w.q()), pool, w.block_tables, np.array([20, 10_000], np.int32), 2,
                            w.scale)
    assert st == oracle.BAD_CTX


def test_workload_generator_shapes():
    for name in ["tiny", "llama3_8b", "llama3_70b", "llama2_7b_int8_prefix", "long_context"]:
        w = named_workload(name)
        assert w.block_tables.shape[0] == w.B
        used = np.concatenate([w.block_tables[b, :w.num_seq_blocks(b)] for b in range(w.B)])
        assert used.min() >= 0 and used.max() < w.num_blocks
    w = named_workload("llama3_70b")
    assert w.unique_blocks() == 16 * 512 and w.num_blocks == math.ceil(1.1 * 8192)
    w = named_workload("long_context")
    assert w.logical_blocks() == 20480
    w = named_workload("llama2_7b_int8_prefix")
    assert w.unique_blocks() < w.logical_blocks()
    assert (w.context_lens >= 2048 + 16).all() and (w.context_lens <= 2048 + 4096).all()
    w = named_workload("llama3_8b")
    assert w.context_lens.min() >= 512 and w.context_lens.max() <= 4096
