"""GPU parity of the shared-prefix decode (pa_decode_opt with share_prefix):
blocks that adjacent sequences share ("LLM 推理底层", "Prefix Caching 与
Copy-on-Write") are attended once per group, and the result must still equal
the oracle's plain decode of every sequence."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import assert_close, gpu_decode, gpu_pool, oracle_full, oracle_one_sequence
from workloads import Geometry, make_workload, named_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def run(w, pool, share=True, num_ctas=0, gen_device="cpu"):
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    out = pa.pa_decode(w.q(gen_device).to(DEV), kc, vc, torch.from_numpy(w.block_tables).to(DEV),
                       torch.from_numpy(w.context_lens).to(DEV), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, num_ctas=num_ctas, share_prefix=share)
    torch.cuda.synchronize()
    return out.float().cpu().numpy(), int(status.item())


def grouped(kv_dtype, d_h, g, groups, prefix, suffix, seed):
    """groups: group id per sequence (-1: none), adjacent members; prefix[i]:
    shared tokens of sequence i's group; suffix[i]: its private tokens."""
    ctx = [p + s for p, s in zip(prefix, suffix)]
    return make_workload("share", Geometry(n_h=2 * g, n_kv=2, d_h=d_h, kv_dtype=kv_dtype), ctx,
                         seed, prefix_len=prefix, group=groups)


CASES = [
    # (dtype, d_h, g, groups, prefix tokens, suffix tokens)
    ("bf16", 128, 4, [0, 0, 0, 1, 1, -1, 2, 2], [256] * 3 + [160] * 2 + [0] + [512] * 2,
     [5, 40, 300, 17, 1, 90, 16, 33]),
    ("int8", 128, 1, [0] * 12, [400] * 12, [3, 17, 50, 9, 100, 1, 64, 31, 7, 260, 44, 2]),
    ("int4", 64, 2, [0, 0, -1, 1, 1, 1], [320, 320, 0, 256, 256, 256], [48, 1, 200, 16, 15, 100]),
    ("bf16", 64, 8, [0, 0, 0, -1, 1, 1], [144] * 3 + [0] + [208] * 2, [20, 16, 1, 77, 3, 400]),
    ("int8", 64, 2, [-1, 0, 0, -1, 1, 1, -1], [0, 128, 128, 0, 512, 512, 0], [30, 2, 19, 0, 60, 8, 5]),
]


@pytest.mark.parametrize("kv_dtype,d_h,g,groups,prefix,suffix", CASES)
def test_shared_prefix_matches_oracle(kv_dtype, d_h, g, groups, prefix, suffix):
    w = grouped(kv_dtype, d_h, g, groups, prefix, suffix, seed=61 + g + d_h)
    pool = gpu_pool(w, DEV, fill_nan=True)
    ref, _ = oracle_full(w)
    plain, st0 = run(w, pool, share=False)
    assert st0 == 0
    for num_ctas in (0, 1, 5, 200):
        out, st = run(w, pool, share=True, num_ctas=num_ctas)
        assert st == 0
        assert_close(out, ref, f"{kv_dtype} d{d_h} g{g} ctas {num_ctas}")
    assert np.abs(out - plain).max() < 2e-2


def test_no_sharing_equals_plain_decode():
    w = make_workload("ns", Geometry(n_h=8, n_kv=2, d_h=128), [300, 17, 1000, 64, 0, 5], seed=71)
    pool = gpu_pool(w, DEV)
    a, _ = run(w, pool, share=False)
    b, st = run(w, pool, share=True)
    assert st == 0 and np.array_equal(a, b)


def test_shared_prefix_full_size_int8_workload():
    # the LLaMA-2-7B INT8 workload: 4 groups of 8 sequences sharing 2048 tokens
    w = named_workload("llama2_7b_int8_prefix")
    pool = gpu_pool(w, DEV, gen_device=DEV)
    out, st = run(w, pool, share=True, gen_device=DEV)
    assert st == 0 and np.isfinite(out).all()
    plain, _ = run(w, pool, share=False, gen_device=DEV)
    assert np.abs(out - plain).max() < 2e-2
    for b in (0, 7, 13, w.B - 1):
        ref, _ = oracle_one_sequence(w, b, gen_device=DEV)
        assert_close(out[b], ref, f"int8 prefix seq {b}")


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8"])
def test_shared_prefix_maximum_batch(kv_dtype):
    # 8192 sequences in runs of 8 sharing 8 full blocks (the shortest prefix
    # that forms a group), ragged suffixes: the detection's largest input and
    # the fused launch's 2 x 8192 units
    rng = np.random.default_rng(6)
    B = 8192
    groups = np.repeat(np.arange(B // 8), 8)
    prefix = np.full(B, 128)
    suffix = rng.integers(1, 50, B)
    w = make_workload("share_maxb", Geometry(n_h=4, n_kv=2, d_h=64, kv_dtype=kv_dtype),
                      (prefix + suffix).tolist(), 17, prefix_len=prefix.tolist(),
                      group=groups.tolist())
    pool = gpu_pool(w, DEV)
    ref, _ = oracle_full(w)
    out, st = run(w, pool, share=True)
    assert st == 0
    assert_close(out, ref, f"{kv_dtype} B=8192 shared")


def test_shared_prefix_too_large_for_the_kernel_decodes_without_sharing():
    # at d_h 128, g = 1, the 2 x 8192 units' prefix arrays do not fit beside
    # the ring: the call decodes without sharing and returns the plain result
    B = 8192
    groups = np.repeat(np.arange(B // 8), 8)
    w = make_workload("share_fallback", Geometry(n_h=2, n_kv=2, d_h=128), [130] * B, 18,
                      prefix_len=[128] * B, group=groups.tolist())
    pool = gpu_pool(w, DEV)
    a, st0 = run(w, pool, share=False)
    b, st1 = run(w, pool, share=True)
    assert st0 == 0 and st1 == 0 and np.array_equal(a, b)
    for s in (0, 4097, B - 1):
        ref, _ = oracle_one_sequence(w, s)
        assert_close(b[s], ref, f"seq {s}")


def detected_groups(w, g, mode=2):
    """(members, shared blocks) of every group pa_share_groups finds."""
    skip, grp, order = pa.pa_share_groups(torch.from_numpy(w.block_tables).to(DEV),
                                          torch.from_numpy(w.context_lens).to(DEV), g, mode)
    torch.cuda.synchronize()
    skip, grp, order = skip.cpu().numpy(), grp.cpu().numpy(), order.cpu().numpy()
    assert sorted(order.tolist()) == list(range(w.B))
    out = []
    for first, n, shared in grp:
        if n == 0:
            break
        members = tuple(int(b) for b in order[first:first + n])
        assert all(skip[b] == shared for b in members)
        out.append((members, int(shared)))
    grouped_seqs = {b for m, _ in out for b in m}
    assert all(skip[b] == 0 for b in range(w.B) if b not in grouped_seqs)
    return out


NON_ADJACENT = [
    # (dtype, d_h, g, groups, prefix tokens, suffix tokens): members of a group
    # are spread over the batch, interleaved with other groups and loners
    ("bf16", 128, 4, [0, 1, 0, -1, 1, 0, 2, 1, 2], [256, 160, 256, 0, 160, 256, 512, 160, 512],
     [5, 40, 300, 17, 1, 90, 16, 33, 7]),
    ("int8", 128, 1, [0, 1] * 6, [400, 256] * 6, [3, 17, 50, 9, 100, 1, 64, 31, 7, 260, 44, 2]),
    ("int4", 64, 2, [1, -1, 0, 1, 0, 1], [256, 0, 320, 256, 320, 256], [48, 1, 200, 16, 15, 100]),
]


@pytest.mark.parametrize("kv_dtype,d_h,g,groups,prefix,suffix", NON_ADJACENT)
def test_shared_prefix_non_adjacent_members(kv_dtype, d_h, g, groups, prefix, suffix):
    # share_prefix=2 finds sharers wherever they sit in the batch; the result
    # equals the oracle's, and so does share_prefix=1's (which groups
    # adjacent sharers only)
    w = grouped(kv_dtype, d_h, g, groups, prefix, suffix, seed=83 + g + d_h)
    pool = gpu_pool(w, DEV, fill_nan=True)
    ref, _ = oracle_full(w)
    plain, st0 = run(w, pool, share=False)
    assert st0 == 0
    out1, st1 = run(w, pool, share=1)
    assert st1 == 0
    assert_close(out1, ref, f"{kv_dtype} d{d_h} g{g} adjacent-only mode")
    for num_ctas in (0, 1, 7, 200):
        out, st = run(w, pool, share=2, num_ctas=num_ctas)
        assert st == 0
        assert_close(out, ref, f"{kv_dtype} d{d_h} g{g} ctas {num_ctas} (non-adjacent)")
    assert np.abs(out - plain).max() < 2e-2
    # the groups found are the workload's: members (by index) and shared blocks
    found = detected_groups(w, g)
    want = {}
    for b, grp in enumerate(groups):
        if grp >= 0:
            want.setdefault(grp, []).append(b)
    assert sorted(found) == sorted((tuple(m), prefix[m[0]] // 16) for m in want.values())


def test_shared_prefix_full_size_int8_workload_shuffled():
    # the LLaMA-2-7B INT8 workload with its 32 sequences in a seeded random
    # order: the 4 groups of 8 are interleaved across the batch
    w = named_workload("llama2_7b_int8_prefix")
    pool = gpu_pool(w, DEV, gen_device=DEV)
    perm = np.random.default_rng(5).permutation(w.B)
    q = w.q(DEV)[torch.from_numpy(perm).to(DEV)]
    bt = torch.from_numpy(np.ascontiguousarray(w.block_tables[perm])).to(DEV)
    cl = torch.from_numpy(np.ascontiguousarray(w.context_lens[perm])).to(DEV)
    kc, vc, ks, vs = pool
    outs = []
    for share in (True, False):
        status = torch.zeros(1, dtype=torch.int32, device=DEV)
        o = pa.pa_decode(q, kc, vc, bt, cl, w.scale, k_scale=ks, v_scale=vs, dev_status=status,
                         share_prefix=2 if share else 0)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        outs.append(o.float().cpu().numpy())
    out, plain = outs
    assert np.isfinite(out).all()
    assert np.abs(out - plain).max() < 2e-2
    # the 4 groups of 8 are found in the shuffled batch, each sharing its 128
    # prefix blocks
    skip, grp, order = pa.pa_share_groups(bt, cl, 1, mode=2)
    torch.cuda.synchronize()
    grp, order = grp.cpu().numpy(), order.cpu().numpy()
    found = sorted(sorted(int(perm[i]) for i in order[f:f + n]) for f, n, s_ in grp if n > 0)
    want = sorted(sorted(np.nonzero(w.group == k)[0].tolist()) for k in range(4))
    assert found == want and all(s_ == 128 for f, n, s_ in grp if n > 0)
    for i in (0, 9, 22, w.B - 1):
        ref, _ = oracle_one_sequence(w, int(perm[i]), gen_device=DEV)
        assert_close(out[i], ref, f"int8 prefix shuffled position {i} (seq {perm[i]})")


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8"])
def test_shared_prefix_maximum_batch_interleaved(kv_dtype):
    # 8192 sequences, 1024 groups of 8 spread over the batch (member j of
    # group k at position j * 1024 + k), share_prefix=2: the detection sorts
    # 8192 keys; every group is found and the output equals the oracle's
    rng = np.random.default_rng(9)
    B = 8192
    groups = np.tile(np.arange(B // 8), 8)
    prefix = np.full(B, 128)
    suffix = rng.integers(1, 50, B)
    w = make_workload("share_maxb_il", Geometry(n_h=4, n_kv=2, d_h=64, kv_dtype=kv_dtype),
                      (prefix + suffix).tolist(), 19, prefix_len=prefix.tolist(),
                      group=groups.tolist())
    pool = gpu_pool(w, DEV)
    ref, _ = oracle_full(w)
    out, st = run(w, pool, share=2)
    assert st == 0
    assert_close(out, ref, f"{kv_dtype} B=8192 interleaved shared")
    found = detected_groups(w, 2)
    assert len(found) == B // 8
    assert all(len(m) == 8 and s == 8 and len({groups[b] for b in m}) == 1 for m, s in found)


def reference_groups(bt, cl, g, mode, min_blocks=8):
    """The grouping rules of pa_share_groups restated in plain Python (lists
    of ints): order, lcp with the previous sequence in that order, runs of
    lcp >= min_blocks cut into chunks of at most gm members."""
    B, max_blocks = bt.shape
    gm = 8 if g <= 2 else 16 // g
    nb = [(int(c) + 15) // 16 if 0 < int(c) <= max_blocks * 16 else 0 for c in cl]

    def fnv(entries):
        h = 2166136261
        for e in entries:
            h = ((h ^ (int(e) & 0xFFFFFFFF)) * 16777619) & 0xFFFFFFFF
        return h

    if mode == 2:
        order = [i for _, i in sorted(
            ((fnv(bt[i, :min_blocks]) if nb[i] > min_blocks else 0xFFFFFFFF), i) for i in range(B))]
    else:
        order = list(range(B))
    lcp = [0] * B
    for p in range(1, B):
        s0, s1 = order[p - 1], order[p]
        lim = max(0, min(nb[s0], nb[s1]) - 1)
        l = 0
        while l < lim and bt[s0, l] == bt[s1, l]:
            l += 1
        lcp[p] = l
    skip, groups = [0] * B, []
    start = 0
    for p in range(B):
        if p == 0 or lcp[p] < min_blocks:
            start = p
        if (p - start) % gm:
            continue
        n, S = 1, None
        while n < gm and p + n < B and lcp[p + n] >= min_blocks:
            S = lcp[p + n] if S is None else min(S, lcp[p + n])
            n += 1
        if n >= 2:
            groups.append((p, n, S))
            for j in range(n):
                skip[order[p + j]] = S
    return skip, groups, order


@pytest.mark.parametrize("mode", [1, 2])
@pytest.mark.parametrize("seed", range(6))
def test_share_groups_match_the_rules(mode, seed):
    # random tables: sequences copy a random partner's leading blocks (3 to
    # 40 of them, so some share fewer than 8), contexts ragged, a few empty
    rng = np.random.default_rng(400 + seed)
    B, max_blocks = int(rng.integers(2, 300)), 64
    g = int(rng.choice([1, 2, 4, 8]))
    bt = rng.permutation(B * max_blocks).reshape(B, max_blocks).astype(np.int32)
    cl = rng.integers(0, max_blocks * 16 + 1, B).astype(np.int32)
    cl[rng.random(B) < 0.05] = 0
    for b in range(1, B):
        if rng.random() < 0.6:
            src = int(rng.integers(0, b))
            k = int(rng.integers(3, 41))
            bt[b, :k] = bt[src, :k]
    skip, grp, order = pa.pa_share_groups(torch.from_numpy(bt).to(DEV), torch.from_numpy(cl).to(DEV),
                                          g, mode)
    torch.cuda.synchronize()
    rskip, rgroups, rorder = reference_groups(bt, cl, g, mode)
    assert order.cpu().numpy().tolist() == rorder
    assert skip.cpu().numpy().tolist() == rskip
    grp = grp.cpu().numpy()
    assert [tuple(int(x) for x in r) for r in grp[:len(rgroups)]] == rgroups
    assert not grp[len(rgroups):].any()
