"""Pure-Python brute force of paged decode attention (TEST INFRASTRUCTURE ONLY).

A second, independent restatement of the computation in plain Python floats
(IEEE double) and nested lists, for tiny inputs. It exists to pin the C oracle:
the two must agree to rounding.

It follows the paged pseudocode of "【infra之路】10-PagedAttention 与 KV Cache
管理" (qwbw.cn) §3.4: for each physical block named by the block table, take
its K rows and score them against the query; softmax over the concatenated
scores; walk the table again and accumulate V weighted by the probabilities.
The score is q.k / sqrt(d) per "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与
PagedAttention 调度" (blog.faulkner.fun), eq. for o_t, with the scale passed in.
"""
from __future__ import annotations

import math
import struct


def bf16_to_float(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def paged_decode_one(q_row, k_blocks, v_blocks, block_table, ctx, scale):
    """One query head.

    q_row: list of floats (d values).
    k_blocks/v_blocks: callables blk -> list of block_size rows (lists of floats)
    for the KV head this query head reads.
    """
    if ctx == 0:
        return [0.0] * len(q_row)
    bs = len(k_blocks(block_table[0]))
    scores = []
    n_blocks = (ctx + bs - 1) // bs
    for i in range(n_blocks):
        rows = k_blocks(block_table[i])
        for o in range(bs):
            if i * bs + o >= ctx:
                break
            scores.append(sum(a * b for a, b in zip(q_row, rows[o])) * scale)
    m = max(scores)
    e = [math.exp(s - m) for s in scores]
    z = sum(e)
    p = [x / z for x in e]
    out = [0.0] * len(q_row)
    j = 0
    for i in range(n_blocks):
        rows = v_blocks(block_table[i])
        for o in range(bs):
            if j >= ctx:
                break
            for d in range(len(out)):
                out[d] += p[j] * rows[o][d]
            j += 1
    return out


def paged_decode(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, n_h, n_kv,
                 scale):
    """q_bits [B][n_h][d] and caches [NB][n_kv][bs][d] of bf16 bit patterns (nested
    sequences or numpy arrays). Returns nested lists [B][n_h][d] of floats."""
    B = len(context_lens)
    g = n_h // n_kv
    out = []
    for b in range(B):
        per_head = []
        for h in range(n_h):
            kv = h // g
            q_row = [bf16_to_float(x) for x in q_bits[b][h]]

            def kb(blk, kv=kv):
                return [[bf16_to_float(x) for x in row] for row in k_cache_bits[blk][kv]]

            def vb(blk, kv=kv):
                return [[bf16_to_float(x) for x in row] for row in v_cache_bits[blk][kv]]

            per_head.append(paged_decode_one(q_row, kb, vb, list(block_tables[b]),
                                             int(context_lens[b]), scale))
        out.append(per_head)
    return out


def attend_rows(q_row, k_rows, v_rows, scale):
    """Softmax attention of one query over an explicit list of K/V rows
    (lists of floats): the plain definition, for the window and sink pins."""
    if not k_rows:
        return [0.0] * len(q_row)
    scores = [sum(a * b for a, b in zip(q_row, k)) * scale for k in k_rows]
    m = max(scores)
    e = [math.exp(s - m) for s in scores]
    z = sum(e)
    out = [0.0] * len(q_row)
    for w, v in zip(e, v_rows):
        for d in range(len(out)):
            out[d] += (w / z) * v[d]
    return out
