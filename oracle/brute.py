"""Pure-Python brute force of paged decode attention (TEST INFRASTRUCTURE ONLY).

A second, independent restatement of the computation in plain Python floats
(IEEE double) and lists, for tiny inputs. It exists to pin the C oracle: the
two must agree to rounding.

It works position by position: logical token j of a sequence is found in
physical block BlockTable[j // bs] at offset j % bs ("LLM 推理底层：KV Cache
显存几何、GQA/MLA 压缩与 PagedAttention 调度", section "逻辑块与物理块映射"), which
gathers the sequence's K and V rows into plain lists; those rows then go
through the attention definition o = softmax(q K^T * scale) V of the same
page (section "自回归解码与 KV Cache 的物理来源", eq. for o_t), with the scale
passed in. Query head h reads KV head h // g (GQA, contiguous groups).
"""
from __future__ import annotations

import math
import struct


def bf16_to_float(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def attend_rows(q_row, k_rows, v_rows, scale):
    """Softmax attention of one query over explicit K/V rows (lists of
    floats); no rows give a zero vector."""
    if not k_rows:
        return [0.0] * len(q_row)
    logits = [scale * sum(a * b for a, b in zip(q_row, k)) for k in k_rows]
    top = max(logits)
    weights = [math.exp(x - top) for x in logits]
    total = sum(weights)
    return [sum(w * v[d] for w, v in zip(weights, v_rows)) / total for d in range(len(q_row))]


def gather_rows(cache_bits, table, ctx, kv_head, block_size):
    """Rows of logical positions 0..ctx-1 of one KV head, through the block
    table, as lists of floats."""
    rows = []
    for j in range(ctx):
        blk = table[j // block_size]
        rows.append([bf16_to_float(x) for x in cache_bits[blk][kv_head][j % block_size]])
    return rows


def paged_decode(q_bits, k_cache_bits, v_cache_bits, block_tables, context_lens, n_h, n_kv,
                 scale):
    """q_bits [B][n_h][d] and caches [NB][n_kv][bs][d] of bf16 bit patterns (nested
    sequences or numpy arrays). Returns nested lists [B][n_h][d] of floats."""
    g = n_h // n_kv
    bs = len(k_cache_bits[0][0])
    out = []
    for b, ctx in enumerate(context_lens):
        table = [int(x) for x in block_tables[b]]
        per_head = []
        for kv in range(n_kv):
            k_rows = gather_rows(k_cache_bits, table, int(ctx), kv, bs)
            v_rows = gather_rows(v_cache_bits, table, int(ctx), kv, bs)
            for h in range(kv * g, (kv + 1) * g):
                q_row = [bf16_to_float(x) for x in q_bits[b][h]]
                per_head.append(attend_rows(q_row, k_rows, v_rows, scale))
        out.append(per_head)
    return out
