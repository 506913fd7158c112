"""Cases shared by the dynamic-range parity tests: workloads whose scores,
K and V magnitudes span the range real caches reach (workloads.PROFILES),
the oracle's answer for them, their closed forms, and the check that the
"rising" profile really makes the running maximum climb."""
import math

import numpy as np

import oracle
from workloads import Geometry, make_workload

PROFILES = ["rising", "v_range", "kv_range", "q_big", "q_small", "q_zero", "same_keys", "onehot"]
POOLS = ["bf16", "int8", "int4"]
HEAD_DIMS = [64, 128]
GROUPS = [1, 8]
CTAS = [0, 1, 300]
CTX = [337, 700, 1201]
WINDOW = 600
LOG2E = 1.0 / math.log(2.0)


def workload(name, seed, kv_dtype, d_h, g, profile, mode):
    geom = Geometry(n_h=2 * g, n_kv=2, d_h=d_h, kv_dtype=kv_dtype)
    kw = dict(profile=profile)
    if profile == "onehot":
        kw["scale"] = 50.0
    ctx = CTX
    if mode == "window":
        kw["window"] = WINDOW
    elif mode == "mq":
        kw["n_q"] = 2 if g == 8 else 4
    elif mode == "share":
        # three sequences share a 320-token prefix (20 whole blocks), one does not
        ctx = [320 + 17, 320 + 400, 320 + 250, 600]
        kw["prefix_len"] = [320, 320, 320, 0]
        kw["group"] = [0, 0, 0, -1]
    return make_workload(name, geom, ctx, seed=seed, **kw)


def run_oracle(w, mode):
    pool = oracle.pool_for(w, fill_nan=True)
    q = oracle.bf16_bits(w.q())
    if mode == "mq":
        ref, st = oracle.decode_mq(q, pool, w.block_tables, w.context_lens, w.geom.n_h, w.scale)
    else:
        ref, st = oracle.decode_window(q, pool, w.block_tables, w.context_lens, w.geom.n_h,
                                       w.scale, window=w.window)
    assert st == 0
    return ref, pool


def dequant_rows(rows, kv_dtype):
    """Dequantised values the pool holds for bf16 rows [n, n_kv, d_h]:
    the rows themselves (bf16), or code * scale formed in fp32 by the
    oracle's quantiser ("kv-cache-guide" §4.2 `dequantize_kv`)."""
    x = rows.float().numpy().astype(np.float64)
    if kv_dtype == "bf16":
        return x
    quant = oracle.quantize_row_int8 if kv_dtype == "int8" else oracle.quantize_row_int4
    bits = oracle.bf16_bits(rows)
    out = np.empty_like(x)
    for t in range(bits.shape[0]):
        for h in range(bits.shape[1]):
            code, sc = quant(bits[t, h])
            out[t, h] = (code.astype(np.float32) * np.float32(sc)).astype(np.float64)
    return out


def closed_form(w, mode):
    """The closed-form output of the q_zero, same_keys and onehot profiles,
    float64 shaped like the decode output, from the workload's rows alone."""
    g = w.geom.g
    n_q = w.n_q
    out = np.zeros((w.B, n_q, w.geom.n_h, w.geom.d_h))
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        _, v = w.seq_kv(b)
        vd = dequant_rows(v, w.geom.kv_dtype)
        for i in range(n_q):
            hi = ctx - n_q + i + 1            # positions [lo, hi) are attended
            lo = max(0, ctx - w.window) if w.window else 0
            if w.profile == "onehot":
                row = vd[ctx - n_q]           # the key 2 * e_k sits at the first new token
            else:
                row = vd[lo:hi].mean(axis=0)
            out[b, i] = np.repeat(row, g, axis=0)
    return out if n_q > 1 else out[:, 0]


def assert_rising(w, pool):
    """Every (sequence, head): over the attended positions, the block maxima
    of the oracle's scores exceed the running maximum of all earlier blocks
    by more than 8 log2 units at least three times."""
    s, st = oracle.scores(oracle.bf16_bits(w.q()), pool, w.block_tables, w.context_lens,
                          w.geom.n_h, w.scale)
    assert st == 0
    for b in range(w.B):
        ctx = int(w.context_lens[b])
        lo = max(0, ctx - w.window) if w.window else 0
        for h in range(w.geom.n_h):
            x = s[b, h, lo:ctx] * LOG2E
            bm = np.array([x[i:i + 16].max() for i in range(0, x.shape[0], 16)])
            climbs = int((bm[1:] > np.maximum.accumulate(bm)[:-1] + 8).sum())
            assert climbs >= 3, (b, h, climbs)
