"""Shared helpers of the GPU tests: fill a device pool through the C ABI and
build the oracle's answer for the same seeded inputs."""
import numpy as np
import torch

import oracle
import paged_kv_cache_94_gb300 as pa

TOL = 1e-2  # |gpu - ref| <= TOL * (1 + |ref|) per output element


def gpu_pool(w, device, gen_device="cpu", fill_nan=False):
    """Device pool holding the workload's history and new tokens, written by
    pa_cache_write. Returns (k_cache, v_cache, k_scale, v_scale)."""
    g = w.geom
    kc, vc, ks, vs = pa.allocate_pool(w.num_blocks, g.n_kv, g.d_h, g.kv_dtype, device)
    if fill_nan:
        if g.kv_dtype == "bf16":
            kc.fill_(float("nan"))
            vc.fill_(float("nan"))
        else:
            ks.fill_(float("nan"))
            vs.fill_(float("nan"))
    for k, v, slots in w.history_chunks(device=gen_device):
        pa.pa_cache_write(k.to(device), v.to(device), torch.from_numpy(slots).to(device), kc, vc,
                          ks, vs)
    kn, vn = w.new_kv(gen_device)
    pa.pa_cache_write(kn.to(device), vn.to(device),
                      torch.from_numpy(w.new_token_slots()).to(device), kc, vc, ks, vs)
    return kc, vc, ks, vs


def gpu_decode(w, pool, device, gen_device="cpu", num_ctas=0, table=None, ctx=None):
    kc, vc, ks, vs = pool
    status = torch.zeros(1, dtype=torch.int32, device=device)
    bt = w.block_tables if table is None else table
    cl = w.context_lens if ctx is None else ctx
    out = pa.pa_decode(w.q(gen_device).to(device), kc, vc, torch.from_numpy(bt).to(device),
                       torch.from_numpy(cl).to(device), w.scale, k_scale=ks, v_scale=vs,
                       dev_status=status, num_ctas=num_ctas)
    torch.cuda.synchronize(device)
    return out, int(status.item())


def oracle_full(w, gen_device="cpu"):
    pool = oracle.pool_for(w, device=gen_device)
    out, st = oracle.decode(oracle.bf16_bits(w.q(gen_device)), pool, w.block_tables,
                            w.context_lens, w.geom.n_h, w.scale)
    assert st == 0
    return out, pool


def oracle_one_sequence(w, b, gen_device="cpu"):
    """Oracle answer for sequence b alone: its rows written into a compact pool
    whose table is 0..nblk-1 (the output does not depend on the physical ids).
    Returns (out [n_h, d_h] float64, compact pool)."""
    g = w.geom
    k, v = w.seq_kv(b, gen_device)
    ctx = int(w.context_lens[b])
    nblk = -(-ctx // g.block_size)
    pool = oracle.Pool(nblk, g.n_kv, g.d_h, g.block_size, g.kv_dtype)
    assert pool.write(oracle.bf16_bits(k), oracle.bf16_bits(v), np.arange(ctx)) == 0
    q = w.q(gen_device)[b:b + 1]
    out, st = oracle.decode(oracle.bf16_bits(q), pool, np.arange(nblk, dtype=np.int32)[None],
                            np.array([ctx], np.int32), g.n_h, w.scale)
    assert st == 0
    return out[0], pool


def assert_close(got, ref, what=""):
    got = np.asarray(got, dtype=np.float64)
    excess = np.abs(got - ref) - TOL * (1.0 + np.abs(ref))
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert (excess <= 0).all(), (f"{what}: max |d| {np.abs(got - ref).max():.3e}, "
                                 f"worst excess {excess.max():.3e}")
    return float(np.abs(got - ref).max())


def pool_bits(t):
    """Device pool tensor -> numpy array of its raw element bits."""
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()
