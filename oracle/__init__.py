"""CPU oracle for paged decode attention (TEST INFRASTRUCTURE ONLY).

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never imports it, and
it never imports the CUDA library: the two share no code. Inputs come from the
``workloads`` generator; expected values come from here.

``oracle/pa_oracle.c`` holds the arithmetic (plain C, double precision for the
attention, fp32 for the INT8 quantiser). ``oracle/brute.py`` is a second,
pure-Python restatement used to pin the C code on tiny inputs.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "pa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

BAD_BLOCK = 1
BAD_SLOT = 2
BAD_CTX = 4


def _stamp() -> str:
    import hashlib
    import platform
    return hashlib.sha256(platform.machine().encode() + open(_SRC, "rb").read()).hexdigest()


def build(force: bool = False) -> str:
    """Compile pa_oracle.c with gcc into oracle/liboracle.so (if stale)."""
    stamp_path = _LIB + ".stamp"
    stamp = _stamp()
    if force or not os.path.exists(_LIB) or not os.path.exists(stamp_path) or \
            open(stamp_path).read() != stamp:
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
        with open(stamp_path, "w") as f:
            f.write(stamp)
    return _LIB


_lib = None


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, dbl = ctypes.c_int32, ctypes.c_int64, ctypes.c_double
        lib.oracle_kv_bytes.restype = dbl
        lib.oracle_kv_bytes.argtypes = [dbl] * 6
        lib.oracle_cache_write_bf16.restype = ctypes.c_int
        lib.oracle_cache_write_bf16.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P]
        lib.oracle_cache_write_int8.restype = ctypes.c_int
        lib.oracle_cache_write_int8.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P, P, P]
        lib.oracle_quantize_row_int8.restype = None
        lib.oracle_quantize_row_int8.argtypes = [P, i32, P, P]
        lib.oracle_cache_write_int4.restype = ctypes.c_int
        lib.oracle_cache_write_int4.argtypes = [P, P, P, i64, i32, i32, i32, i64, P, P, P, P]
        lib.oracle_quantize_row_int4.restype = None
        lib.oracle_quantize_row_int4.argtypes = [P, i32, P, P]
        lib.oracle_decode.restype = ctypes.c_int
        lib.oracle_decode.argtypes = [P, P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32, i64,
                                      dbl, P]
        lib.oracle_decode_mq.restype = ctypes.c_int
        lib.oracle_decode_mq.argtypes = [P, P, P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32,
                                         i32, i64, dbl, P]
        lib.oracle_decode_window.restype = ctypes.c_int
        lib.oracle_decode_window.argtypes = [P, P, P, P, P, i32, P, i32, P, i32, i32, i32, i32,
                                             i32, i64, dbl, i32, i32, P, P, P]
        lib.oracle_scores.restype = ctypes.c_int
        lib.oracle_scores.argtypes = [P, P, P, i32, P, i32, P, i32, i32, i32, i32, i32, i64, dbl,
                                      i64, P]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (on any device)."""
    import torch
    assert t.dtype == torch.bfloat16
    return np.ascontiguousarray(t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16))


def kv_bytes(L, n_kv, d_h, S, B, b_dtype) -> float:
    """M_KV = 2 L n_kv d_h S B b_dtype (bytes of K and V over all layers)."""
    return _load().oracle_kv_bytes(float(L), float(n_kv), float(d_h), float(S), float(B), float(b_dtype))


class Pool:
    """A paged K/V pool held by the oracle: [num_blocks, n_kv, block_size, d_h]."""

    def __init__(self, num_blocks: int, n_kv: int, d_h: int, block_size: int = 16,
                 kv_dtype: str = "bf16", fill_nan: bool = False):
        self.num_blocks, self.n_kv, self.d_h, self.block_size = num_blocks, n_kv, d_h, block_size
        self.kv_dtype = kv_dtype
        shape = (num_blocks, n_kv, block_size, d_h)
        if kv_dtype == "bf16":
            fill = 0x7FC0 if fill_nan else 0  # bf16 quiet NaN
            self.k = np.full(shape, fill, dtype=np.uint16)
            self.v = np.full(shape, fill, dtype=np.uint16)
            self.k_scale = self.v_scale = None
        elif kv_dtype in ("int8", "int4"):
            if kv_dtype == "int8":
                self.k = np.full(shape, 0, dtype=np.int8)
                self.v = np.full(shape, 0, dtype=np.int8)
            else:  # two codes per byte
                self.k = np.full(shape[:3] + (d_h // 2,), 0, dtype=np.uint8)
                self.v = np.full(shape[:3] + (d_h // 2,), 0, dtype=np.uint8)
            sfill = np.nan if fill_nan else 0.0
            self.k_scale = np.full(shape[:3], sfill, dtype=np.float32)
            self.v_scale = np.full(shape[:3], sfill, dtype=np.float32)
        else:
            raise ValueError(kv_dtype)

    def write(self, k_bits: np.ndarray, v_bits: np.ndarray, slots: np.ndarray) -> int:
        """Append rows k/v (uint16 bf16 bits [T, n_kv, d_h]) at the given slots."""
        lib = _load()
        k_bits = np.ascontiguousarray(k_bits, dtype=np.uint16)
        v_bits = np.ascontiguousarray(v_bits, dtype=np.uint16)
        slots = np.ascontiguousarray(slots, dtype=np.int64)
        T = slots.shape[0]
        assert k_bits.shape == (T, self.n_kv, self.d_h) and v_bits.shape == k_bits.shape
        if self.kv_dtype == "bf16":
            return lib.oracle_cache_write_bf16(_ptr(k_bits), _ptr(v_bits), _ptr(slots), T, self.n_kv,
                                               self.d_h, self.block_size, self.num_blocks,
                                               _ptr(self.k), _ptr(self.v))
        fn = lib.oracle_cache_write_int8 if self.kv_dtype == "int8" else lib.oracle_cache_write_int4
        return fn(_ptr(k_bits), _ptr(v_bits), _ptr(slots), T, self.n_kv, self.d_h,
                  self.block_size, self.num_blocks, _ptr(self.k), _ptr(self.v),
                  _ptr(self.k_scale), _ptr(self.v_scale))

    def decode(self, q_bits: np.ndarray, block_tables: np.ndarray, context_lens: np.ndarray,
               n_h: int, scale: float) -> tuple[np.ndarray, int]:
        """Decode attention for every sequence and head: float64 [B, n_h, d_h] and status."""
        return decode(q_bits, self, block_tables, context_lens, n_h, scale)


KV_KIND = {"bf16": 0, "int8": 1, "int4": 2}


def quantize_row_int4(x_bits: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """Quantise one bf16 row (uint16 bits) -> (INT4 codes, one per int8, fp32 scale)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    code = np.zeros(x_bits.shape[0], dtype=np.int8)
    sc = np.zeros(1, dtype=np.float32)
    _load().oracle_quantize_row_int4(_ptr(x_bits), x_bits.shape[0], _ptr(code), _ptr(sc))
    return code, sc[0]


def quantize_row_int8(x_bits: np.ndarray) -> tuple[np.ndarray, np.float32]:
    """Quantise one bf16 row (uint16 bits) -> (int8 codes, fp32 scale)."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    code = np.zeros(x_bits.shape[0], dtype=np.int8)
    sc = np.zeros(1, dtype=np.float32)
    _load().oracle_quantize_row_int8(_ptr(x_bits), x_bits.shape[0], _ptr(code), _ptr(sc))
    return code, sc[0]


def decode(q_bits: np.ndarray, pool: Pool, block_tables: np.ndarray, context_lens: np.ndarray,
           n_h: int, scale: float) -> tuple[np.ndarray, int]:
    lib = _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = ctx.shape[0]
    assert q_bits.shape == (B, n_h, pool.d_h)
    out = np.zeros((B, n_h, pool.d_h), dtype=np.float64)
    st = lib.oracle_decode(_ptr(q_bits), _ptr(pool.k), _ptr(pool.v), _ptr(pool.k_scale),
                           _ptr(pool.v_scale), KV_KIND[pool.kv_dtype], _ptr(bt),
                           bt.shape[1], _ptr(ctx), B, n_h, pool.n_kv, pool.d_h, pool.block_size,
                           pool.num_blocks, float(scale), _ptr(out))
    return out, st


def scores(q_bits: np.ndarray, pool: Pool, block_tables: np.ndarray, context_lens: np.ndarray,
           n_h: int, scale: float) -> tuple[np.ndarray, int]:
    """Raw scores scale * <q_h, K_j>: float64 [B, n_h, max ctx] (NaN past a
    sequence's context) and status."""
    lib = _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = ctx.shape[0]
    assert q_bits.shape == (B, n_h, pool.d_h)
    max_ctx = max(int(ctx.max()) if B else 0, 1)
    out = np.zeros((B, n_h, max_ctx), dtype=np.float64)
    st = lib.oracle_scores(_ptr(q_bits), _ptr(pool.k), _ptr(pool.k_scale), KV_KIND[pool.kv_dtype],
                           _ptr(bt), bt.shape[1], _ptr(ctx), B, n_h, pool.n_kv, pool.d_h,
                           pool.block_size, pool.num_blocks, float(scale), max_ctx, _ptr(out))
    return out, st


def decode_window(q_bits: np.ndarray, pool: Pool, block_tables: np.ndarray,
                  context_lens: np.ndarray, n_h: int, scale: float, window: int = 0,
                  n_sink: int = 0, sink_k_bits: Optional[np.ndarray] = None,
                  sink_v_bits: Optional[np.ndarray] = None) -> tuple[np.ndarray, int]:
    """Decode attention over the last `window` tokens (0 = all), with the
    first n_sink positions read from bf16 sink rows [B, n_kv, n_sink, d_h]
    (INT8 pools only). float64 [B, n_h, d_h] and status."""
    lib = _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    B = ctx.shape[0]
    assert q_bits.shape == (B, n_h, pool.d_h)
    if n_sink:
        assert pool.kv_dtype in ("int8", "int4")
        sink_k_bits = np.ascontiguousarray(sink_k_bits, dtype=np.uint16)
        sink_v_bits = np.ascontiguousarray(sink_v_bits, dtype=np.uint16)
        assert sink_k_bits.shape == (B, pool.n_kv, n_sink, pool.d_h)
        assert sink_v_bits.shape == sink_k_bits.shape
    else:
        sink_k_bits = sink_v_bits = None
    out = np.zeros((B, n_h, pool.d_h), dtype=np.float64)
    st = lib.oracle_decode_window(_ptr(q_bits), _ptr(pool.k), _ptr(pool.v), _ptr(pool.k_scale),
                                  _ptr(pool.v_scale), KV_KIND[pool.kv_dtype],
                                  _ptr(bt), bt.shape[1], _ptr(ctx), B, n_h, pool.n_kv, pool.d_h,
                                  pool.block_size, pool.num_blocks, float(scale), int(window),
                                  int(n_sink), _ptr(sink_k_bits), _ptr(sink_v_bits), _ptr(out))
    return out, st


def decode_mq(q_bits: np.ndarray, pool: Pool, block_tables: np.ndarray,
              context_lens: np.ndarray, n_h: int, scale: float) -> tuple[np.ndarray, int]:
    """Multi-query decode: q [B, n_q, n_h, d_h] (bf16 bits), the last n_q
    positions of each sequence attending causally. float64 [B, n_q, n_h, d_h]."""
    lib = _load()
    q_bits = np.ascontiguousarray(q_bits, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    ctx = np.ascontiguousarray(context_lens, dtype=np.int32)
    B, n_q = q_bits.shape[:2]
    assert q_bits.shape == (B, n_q, n_h, pool.d_h) and ctx.shape == (B,)
    out = np.zeros(q_bits.shape, dtype=np.float64)
    st = lib.oracle_decode_mq(_ptr(q_bits), _ptr(pool.k), _ptr(pool.v), _ptr(pool.k_scale),
                              _ptr(pool.v_scale), KV_KIND[pool.kv_dtype], _ptr(bt), bt.shape[1],
                              _ptr(ctx), B, n_q, n_h, pool.n_kv, pool.d_h, pool.block_size,
                              pool.num_blocks, float(scale), _ptr(out))
    return out, st


def pool_for(workload, seqs=None, fill_nan: bool = False, include_new: bool = True,
             device="cpu") -> Pool:
    """Oracle pool holding the workload's history (and, by default, the new tokens).

    seqs restricts the pool contents to those sequences (the rest stays at the
    fill value); the pool keeps the workload's full physical size.
    """
    g = workload.geom
    pool = Pool(workload.num_blocks, g.n_kv, g.d_h, g.block_size, g.kv_dtype, fill_nan=fill_nan)
    for k, v, slots in workload.history_chunks(device=device, seqs=seqs):
        st = pool.write(bf16_bits(k), bf16_bits(v), slots)
        assert st == 0
    if include_new:
        kn, vn = workload.new_kv(device=device)
        slots = workload.new_token_slots()
        if seqs is not None:
            mask = np.zeros(workload.B, bool)
            mask[list(seqs)] = True
            slots = np.where(mask, slots, -1)
        st = pool.write(bf16_bits(kn), bf16_bits(vn), slots)
        assert st == 0
    return pool
