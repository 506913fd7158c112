"""Python binding of libpa.so: paged KV-cache decode attention on GB300.

Argument marshalling only. Every step of the computation runs in the CUDA
kernels of libpa.so (see include/pa.h for the C ABI); this module checks the
torch tensors it is given, passes their device pointers and the current CUDA
stream, and raises PAError on a non-OK status. There is no CPU fallback: if
the library has not been built, or no CUDA device is present, the calls raise.

    pa_cache_write(k, v, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None)
    out = pa_decode(q, k_cache, v_cache, block_tables, context_lens, scale,
                    k_scale=None, v_scale=None)
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "lib", "libpa.so")

PA_KV_BF16 = 0
PA_KV_INT8 = 1
PA_KV_INT4 = 2

PA_DEV_BAD_BLOCK = 0x1
PA_DEV_BAD_SLOT = 0x2
PA_DEV_BAD_CONTEXT = 0x4
PA_DEV_TIMEOUT = 0x8

STATUS = {
    0: "PA_OK", -1: "PA_ERR_NULL", -2: "PA_ERR_SHAPE", -3: "PA_ERR_DTYPE",
    -4: "PA_ERR_UNSUPPORTED", -5: "PA_ERR_BAD_BLOCK", -6: "PA_ERR_BAD_SLOT",
    -7: "PA_ERR_WORKSPACE", -8: "PA_ERR_CUDA", -9: "PA_ERR_BAD_CONTEXT",
    -10: "PA_ERR_TIMEOUT", -11: "PA_ERR_ALIGNMENT", -12: "PA_ERR_OUT_OF_BLOCKS",
    -13: "PA_ERR_STATE",
}
PA_ERR_OUT_OF_BLOCKS = -12
PA_ERR_STATE = -13
EXPORTED = ["pa_cache_write", "pa_decode_workspace_size", "pa_decode_workspace_init",
            "pa_decode", "pa_decode_ex", "pa_decode_noalloc", "pa_decode_default_ctas",
            "pa_plan_owner", "pa_block_copy", "pa_decode_opt", "pa_sink_write",
            "pa_decode_mq", "pa_decode_mq_ex", "pa_decode_mq_workspace_size", "pa_decode_opt_workspace_size",
            "pa_status_string", "pa_status_from_device", "pa_version", "pa_wait_selftest",
            "pa_kv_read_probe", "pa_share_groups",
            # host block manager (include/pa_alloc.h)
            "pa_allocator_create", "pa_allocator_destroy", "pa_allocator_allocate_prompt",
            "pa_allocator_append_slots", "pa_allocator_fork", "pa_allocator_free",
            "pa_allocator_num_free", "pa_allocator_block_info", "pa_allocator_free_order",
            "pa_block_hash"]


class PAError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        msg = _lib().pa_status_string(status).decode() if _LIB is not None else STATUS.get(status)
        super().__init__(f"{where}: {msg} ({status})" if where else f"{msg} ({status})")


class pa_geom(ctypes.Structure):
    _fields_ = [("num_blocks", ctypes.c_int64), ("n_h", ctypes.c_int32),
                ("n_kv", ctypes.c_int32), ("d_h", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("kv_dtype", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class pa_decode_opts(ctypes.Structure):
    _fields_ = [("window", ctypes.c_int32), ("n_sink", ctypes.c_int32),
                ("sink_k", ctypes.c_void_p), ("sink_v", ctypes.c_void_p),
                ("num_ctas", ctypes.c_int32), ("share_prefix", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


_LIB = None
_LIB_LOCK = threading.Lock()


def _lib():
    """Load libpa.so (raises if it was not built)."""
    global _LIB
    if _LIB is not None:
        return _LIB
    with _LIB_LOCK:
        if _LIB is not None:
            return _LIB
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                f"g.build()'` (nvcc, sm_103a). There is no CPU fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        P, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        lib.pa_cache_write.restype = ctypes.c_int
        lib.pa_cache_write.argtypes = [P, P, P, i64, P, P, P, P, pa_geom, P, P]
        lib.pa_decode_workspace_size.restype = sz
        lib.pa_decode_workspace_size.argtypes = [pa_geom, i32, i32]
        lib.pa_decode_workspace_init.restype = ctypes.c_int
        lib.pa_decode_workspace_init.argtypes = [P, sz, P]
        dec = [P, P, P, P, P, P, i32, P, i32, f32, P, P, sz, pa_geom, P, P]
        lib.pa_decode.restype = ctypes.c_int
        lib.pa_decode.argtypes = dec
        lib.pa_decode_ex.restype = ctypes.c_int
        lib.pa_decode_ex.argtypes = dec + [i32]
        lib.pa_decode_noalloc.restype = ctypes.c_int
        lib.pa_decode_noalloc.argtypes = [P, P, P, P, P, P, i32, P, i32, f32, P, pa_geom, P, P]
        lib.pa_decode_default_ctas.restype = i32
        lib.pa_decode_default_ctas.argtypes = [pa_geom, i32]
        lib.pa_plan_owner.restype = i32
        lib.pa_plan_owner.argtypes = [i64, i64, i32]
        lib.pa_status_string.restype = ctypes.c_char_p
        lib.pa_status_string.argtypes = [ctypes.c_int]
        lib.pa_status_from_device.restype = ctypes.c_int
        lib.pa_status_from_device.argtypes = [i32]
        lib.pa_version.restype = i32
        lib.pa_version.argtypes = []
        lib.pa_wait_selftest.restype = ctypes.c_int
        lib.pa_wait_selftest.argtypes = [P, i32, P]
        lib.pa_decode_mq.restype = ctypes.c_int
        lib.pa_decode_mq.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, f32, P, P, sz, pa_geom,
                                     P, P]
        lib.pa_decode_mq_ex.restype = ctypes.c_int
        lib.pa_decode_mq_ex.argtypes = lib.pa_decode_mq.argtypes + [i32]
        lib.pa_decode_mq_workspace_size.restype = sz
        lib.pa_decode_mq_workspace_size.argtypes = [pa_geom, i32, i32, i32]
        lib.pa_decode_opt_workspace_size.restype = sz
        lib.pa_decode_opt_workspace_size.argtypes = [pa_geom, i32, P]
        lib.pa_decode_opt.restype = ctypes.c_int
        lib.pa_decode_opt.argtypes = dec[:14] + [P] + dec[14:]
        lib.pa_sink_write.restype = ctypes.c_int
        lib.pa_sink_write.argtypes = [P, P, P, P, i64, P, P, i32, i32, pa_geom, P]
        lib.pa_kv_read_probe.restype = ctypes.c_int
        lib.pa_kv_read_probe.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, P, pa_geom, P]
        lib.pa_share_groups.restype = ctypes.c_int
        lib.pa_share_groups.argtypes = [P, i32, P, i32, i32, i32, P, P, P, P]
        lib.pa_block_copy.restype = ctypes.c_int
        lib.pa_block_copy.argtypes = [P, P, P, P, P, i32, pa_geom, P, P]
        u64 = ctypes.c_uint64
        lib.pa_allocator_create.restype = ctypes.c_int
        lib.pa_allocator_create.argtypes = [i64, i32, ctypes.POINTER(P)]
        lib.pa_allocator_destroy.restype = None
        lib.pa_allocator_destroy.argtypes = [P]
        lib.pa_allocator_allocate_prompt.restype = ctypes.c_int
        lib.pa_allocator_allocate_prompt.argtypes = [P, P, i32, P, i32, P, P]
        lib.pa_allocator_append_slots.restype = ctypes.c_int
        lib.pa_allocator_append_slots.argtypes = [P, P, i32, P, P, i32, P, P, P, P]
        lib.pa_allocator_fork.restype = ctypes.c_int
        lib.pa_allocator_fork.argtypes = [P, P, i32]
        lib.pa_allocator_free.restype = ctypes.c_int
        lib.pa_allocator_free.argtypes = [P, P, i32]
        lib.pa_allocator_num_free.restype = i64
        lib.pa_allocator_num_free.argtypes = [P]
        lib.pa_allocator_block_info.restype = ctypes.c_int
        lib.pa_allocator_block_info.argtypes = [P, i64, P, P, P, P]
        lib.pa_allocator_free_order.restype = ctypes.c_int
        lib.pa_allocator_free_order.argtypes = [P, P, i64, P]
        lib.pa_block_hash.restype = u64
        lib.pa_block_hash.argtypes = [u64, P, i32]
        _LIB = lib
        return lib


def library():
    """The loaded ctypes library (for direct C-ABI calls)."""
    return _lib()


def _check(status: int, where: str):
    if status != 0:
        raise PAError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_ptr(stream) -> Optional[int]:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def pa_wait_selftest(dev_status: torch.Tensor, limit_us: int = 2000, stream=None) -> None:
    """Run the bounded-wait self-test: a wait on a barrier nothing arrives on
    gives up after limit_us and sets PA_DEV_TIMEOUT in dev_status (int32, device)."""
    _need_cuda("dev_status", dev_status, torch.int32)
    _check(_lib().pa_wait_selftest(_ptr(dev_status), int(limit_us), _stream_ptr(stream)),
           "pa_wait_selftest")


class Prepared:
    """One validated library call with its arguments marshalled, issued again
    by calling it: for a serving loop that repeats the same call on the same
    buffers (the tensors' contents may change, not their addresses or shapes).
    The stream is the one given at preparation, else the current stream at
    each call. Returns what the unprepared call returns (the output tensor)."""

    __slots__ = ("_fn", "_args", "_si", "_what", "_result", "_stream")

    def __init__(self, fn, args, stream_index, what, result, stream):
        self._fn, self._args, self._si = fn, list(args), stream_index
        self._what, self._result, self._stream = what, result, stream

    def __call__(self):
        self._args[self._si] = _stream_ptr(self._stream)
        st = self._fn(*self._args)
        if st != 0:
            raise PAError(st, self._what)
        return self._result


def _need_cuda(name: str, t: torch.Tensor, dtype=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")


def geometry(k_cache: torch.Tensor, n_h: int) -> pa_geom:
    """pa_geom of a pool [num_blocks, n_kv, 16, d_h] (bf16 or int8; uint8 [.., d_h/2]
    for INT4) for n_h query heads."""
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be [num_blocks, n_kv, block_size, d_h]")
    nb, n_kv, bs, d = k_cache.shape
    if k_cache.dtype == torch.bfloat16:
        dt = PA_KV_BF16
    elif k_cache.dtype == torch.int8:
        dt = PA_KV_INT8
    elif k_cache.dtype == torch.uint8:
        dt = PA_KV_INT4  # two codes per byte
        d = 2 * d
    else:
        raise TypeError("k_cache must be bfloat16, int8 or uint8 (INT4)")
    return pa_geom(num_blocks=nb, n_h=n_h, n_kv=n_kv, d_h=d, block_size=bs, kv_dtype=dt, reserved=0)


def pa_cache_write(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                   k_cache: torch.Tensor, v_cache: torch.Tensor,
                   k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                   dev_status: Optional[torch.Tensor] = None, stream=None,
                   prepare: bool = False):
    """Append rows k, v [T, n_kv, d_h] (bf16) at slot_mapping [T] (int64) into the pool.
    prepare=True validates and returns a Prepared call instead of running it."""
    _need_cuda("k", k, torch.bfloat16)
    _need_cuda("v", v, torch.bfloat16)
    _need_cuda("slot_mapping", slot_mapping, torch.int64)
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    g = geometry(k_cache, n_h=k_cache.shape[1])
    if k.shape != (slot_mapping.shape[0], g.n_kv, g.d_h) or v.shape != k.shape:
        raise ValueError("k, v must be [num_tokens, n_kv, d_h] matching the pool and slot_mapping")
    if g.kv_dtype != PA_KV_BF16:
        for nm, s in (("k_scale", k_scale), ("v_scale", v_scale)):
            if s is None:
                raise ValueError(f"{nm} is required for an int8/int4 pool")
            _need_cuda(nm, s, torch.float32)
            if tuple(s.shape) != tuple(k_cache.shape[:3]):
                raise ValueError(f"{nm} must be [num_blocks, n_kv, block_size]")
    if dev_status is not None:
        _need_cuda("dev_status", dev_status, torch.int32)
    call = Prepared(_lib().pa_cache_write,
                    [_ptr(k), _ptr(v), _ptr(slot_mapping), slot_mapping.shape[0], _ptr(k_cache),
                     _ptr(v_cache), _ptr(k_scale), _ptr(v_scale), g, _ptr(dev_status), None],
                    10, "pa_cache_write", None, stream)
    return call if prepare else call()


_WS: dict = {}
_WS_SIZES: dict = {}
_WS_LOCK = threading.Lock()


def _counter_bytes(g: pa_geom, num_seqs: int, share_prefix: bool = False) -> int:
    """Leading workspace bytes that must be zero on entry (the library leaves
    them zero): the unit counters (a shared-prefix call has 2 * num_seqs
    units per kv head: the groups, then the sequences)."""
    n = 2 * num_seqs * g.n_kv if share_prefix else num_seqs * g.n_kv
    return (4 * n + 255) // 256 * 256


def decode_workspace(g: pa_geom, num_seqs: int, device: torch.device, num_ctas: int = 0,
                     stream=None, n_q: int = 1, share_prefix: bool = False) -> torch.Tensor:
    """A workspace for pa_decode, cached per device.

    Its leading counter area must be zero on entry; pa_decode leaves it zero,
    so the cache only re-zeroes it when a call needs a larger counter area
    than the buffer has had zeroed so far.
    """
    key = device.index if device.index is not None else torch.cuda.current_device()
    size_key = (key, g.num_blocks, g.n_h, g.n_kv, g.d_h, g.kv_dtype, num_seqs, num_ctas, n_q,
                share_prefix)
    nbytes = _WS_SIZES.get(size_key)
    if nbytes is None:
        if share_prefix:
            o = pa_decode_opts(num_ctas=int(num_ctas), share_prefix=1)
            nbytes = _lib().pa_decode_opt_workspace_size(g, num_seqs, ctypes.byref(o))
        elif n_q == 1:
            nbytes = _lib().pa_decode_workspace_size(g, num_seqs, num_ctas)
        else:
            nbytes = _lib().pa_decode_mq_workspace_size(g, num_seqs, n_q, num_ctas)
        if nbytes == 0:
            raise PAError(-4 if n_q > 1 else -2, "pa_decode_workspace_size")
        _WS_SIZES[size_key] = nbytes
    need_zero = _counter_bytes(g, num_seqs, share_prefix)
    with _WS_LOCK:
        ent = _WS.get(key)
        if ent is None or ent[0].numel() < nbytes:
            ws = torch.zeros(max(nbytes, 1 << 20), dtype=torch.uint8, device=device)
            ent = [ws, ws.numel()]
            _WS[key] = ent
        elif ent[1] < need_zero:
            s = torch.cuda.current_stream(device) if stream is None else stream
            _check(_lib().pa_decode_workspace_init(_ptr(ent[0]), ent[0].numel(),
                                                   ctypes.c_void_p(s.cuda_stream)),
                   "pa_decode_workspace_init")
            ent[1] = ent[0].numel()
        # after this call only the counter area is known to be zero: the rest
        # is scratch, where a later call with more units puts its counters
        ent[1] = need_zero
        return ent[0]


def pa_decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
              out: Optional[torch.Tensor] = None, k_scale: Optional[torch.Tensor] = None,
              v_scale: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
              dev_status: Optional[torch.Tensor] = None, stream=None, num_ctas: int = 0,
              window: int = 0, sink_k: Optional[torch.Tensor] = None,
              sink_v: Optional[torch.Tensor] = None, share_prefix: int = 0,
              prepare: bool = False):
    """Decode attention: q [B, n_h, d_h] bf16 over the paged pool -> out [B, n_h, d_h] bf16.

    block_tables [B, max_blocks] int32 and context_lens [B] int32 live on the device.
    num_ctas > 0 forces the number of CTAs the work is split over (pa_decode_ex).
    window > 0 attends the last `window` tokens of each sequence; sink_k/sink_v
    (bf16 [B, n_kv, n_sink, d_h], INT8 pools) hold the unquantised rows of the
    first n_sink positions (pa_decode_opt). share_prefix (True or 1: sharers
    adjacent in the batch; 2: anywhere) attends blocks that sequences share
    once per group (pa_decode_opt, share_prefix).
    prepare=True validates and returns a Prepared call instead of running it.
    """
    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if q.dim() != 3:
        raise ValueError("q must be [num_seqs, n_h, d_h]")
    B, n_h, d = q.shape
    g = geometry(k_cache, n_h)
    if d != g.d_h or block_tables.dim() != 2 or block_tables.shape[0] != B or \
            context_lens.shape != (B,):
        raise ValueError("q, block_tables, context_lens disagree on num_seqs or d_h")
    if g.kv_dtype != PA_KV_BF16:
        for nm, s in (("k_scale", k_scale), ("v_scale", v_scale)):
            if s is None:
                raise ValueError(f"{nm} is required for an int8/int4 pool")
            _need_cuda(nm, s, torch.float32)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, torch.bfloat16)
        if out.shape != q.shape:
            raise ValueError("out must have the shape of q")
    if workspace is None:
        workspace = decode_workspace(g, B, q.device, num_ctas, stream,
                                     share_prefix=bool(share_prefix))
    else:
        _need_cuda("workspace", workspace)
    if dev_status is not None:
        _need_cuda("dev_status", dev_status, torch.int32)
    lib = _lib()
    args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, float(scale),
            _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size(), g,
            _ptr(dev_status), _stream_ptr(stream)]
    if window or sink_k is not None or sink_v is not None or share_prefix:
        n_sink = 0
        if sink_k is not None or sink_v is not None:
            _need_cuda("sink_k", sink_k, torch.bfloat16)
            _need_cuda("sink_v", sink_v, torch.bfloat16)
            n_sink = sink_k.shape[2]
            if sink_k.shape != (B, g.n_kv, n_sink, g.d_h) or sink_v.shape != sink_k.shape:
                raise ValueError("sink_k, sink_v must be [num_seqs, n_kv, n_sink, d_h]")
        opts = pa_decode_opts(window=int(window), n_sink=n_sink, sink_k=_ptr(sink_k),
                              sink_v=_ptr(sink_v), num_ctas=int(num_ctas),
                              share_prefix=int(share_prefix), reserved=0)
        call = Prepared(lib.pa_decode_opt, args[:14] + [ctypes.byref(opts)] + args[14:], 16,
                        "pa_decode", out, stream)
    elif num_ctas > 0:
        call = Prepared(lib.pa_decode_ex, args + [int(num_ctas)], 15, "pa_decode", out, stream)
    else:
        call = Prepared(lib.pa_decode, args, 15, "pa_decode", out, stream)
    return call if prepare else call()


def pa_decode_mq(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 block_tables: torch.Tensor, context_lens: torch.Tensor, scale: float,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 dev_status: Optional[torch.Tensor] = None, stream=None,
                 k_scale: Optional[torch.Tensor] = None,
                 v_scale: Optional[torch.Tensor] = None, prepare: bool = False,
                 num_ctas: int = 0):
    """Multi-query decode: q [B, n_q, n_h, d_h] bf16 (the last n_q tokens of each
    sequence, attending causally) over a bf16, INT8 or INT4 pool (scales as
    pa_decode's) -> out of q's shape. num_ctas > 0 forces the CTA count
    (pa_decode_mq_ex). prepare=True returns a Prepared call."""
    _need_cuda("q", q, torch.bfloat16)
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    if q.dim() != 4:
        raise ValueError("q must be [num_seqs, n_q, n_h, d_h]")
    B, n_q, n_h, d = q.shape
    g = geometry(k_cache, n_h)
    if d != g.d_h or block_tables.dim() != 2 or block_tables.shape[0] != B or \
            context_lens.shape != (B,):
        raise ValueError("q, block_tables, context_lens disagree on num_seqs or d_h")
    if g.kv_dtype != PA_KV_BF16:
        for nm, s in (("k_scale", k_scale), ("v_scale", v_scale)):
            if s is None:
                raise ValueError(f"{nm} is required for an int8/int4 pool")
            _need_cuda(nm, s, torch.float32)
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, torch.bfloat16)
        if out.shape != q.shape:
            raise ValueError("out must have the shape of q")
    if workspace is None:
        workspace = decode_workspace(g, B, q.device, num_ctas, stream, n_q=n_q)
    else:
        _need_cuda("workspace", workspace)
    if dev_status is not None:
        _need_cuda("dev_status", dev_status, torch.int32)
    args = [_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
            _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, n_q,
            float(scale), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size(), g, _ptr(dev_status), None]
    if num_ctas > 0:
        call = Prepared(_lib().pa_decode_mq_ex, args + [int(num_ctas)], 16, "pa_decode_mq", out,
                        stream)
    else:
        call = Prepared(_lib().pa_decode_mq, args, 16, "pa_decode_mq", out, stream)
    return call if prepare else call()


def pa_sink_write(k: torch.Tensor, v: torch.Tensor, seq_rows: torch.Tensor,
                  positions: torch.Tensor, sink_k: torch.Tensor, sink_v: torch.Tensor,
                  stream=None) -> None:
    """Store the bf16 rows of tokens at positions < n_sink into the sink rows
    sink_k/sink_v [num_seqs, n_kv, n_sink, d_h] (seq_rows, positions: int32 [T])."""
    _need_cuda("k", k, torch.bfloat16)
    _need_cuda("v", v, torch.bfloat16)
    _need_cuda("seq_rows", seq_rows, torch.int32)
    _need_cuda("positions", positions, torch.int32)
    _need_cuda("sink_k", sink_k, torch.bfloat16)
    _need_cuda("sink_v", sink_v, torch.bfloat16)
    if sink_k.dim() != 4 or sink_v.shape != sink_k.shape:
        raise ValueError("sink_k, sink_v must be [num_seqs, n_kv, n_sink, d_h]")
    B, n_kv, n_sink, d = sink_k.shape
    T = k.shape[0]
    if k.shape != (T, n_kv, d) or v.shape != k.shape or seq_rows.shape != (T,) or \
            positions.shape != (T,):
        raise ValueError("k, v [T, n_kv, d_h], seq_rows and positions [T] must agree")
    g = pa_geom(num_blocks=1, n_h=n_kv, n_kv=n_kv, d_h=d, block_size=16, kv_dtype=PA_KV_INT8,
                reserved=0)
    _check(_lib().pa_sink_write(_ptr(k), _ptr(v), _ptr(seq_rows), _ptr(positions), T,
                                _ptr(sink_k), _ptr(sink_v), n_sink, B, g, _stream_ptr(stream)),
           "pa_sink_write")


def pa_kv_read_probe(k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, n_h: int, heads_per_read: int, num_ctas: int,
                     sink: torch.Tensor, k_scale: Optional[torch.Tensor] = None,
                     v_scale: Optional[torch.Tensor] = None, stream=None) -> None:
    """Read the K/V bytes a decode of this batch reads, with plain loads and
    no arithmetic (a measurement aid); sink: uint8/int32 tensor of >= 4 *
    num_ctas bytes, written."""
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    _need_cuda("sink", sink)
    if sink.numel() * sink.element_size() < 4 * num_ctas:
        raise ValueError("sink must hold num_ctas uint32 words")
    g = geometry(k_cache, n_h)
    s = torch.cuda.current_stream(k_cache.device) if stream is None else stream
    _check(_lib().pa_kv_read_probe(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                                   _ptr(block_tables), block_tables.shape[1], _ptr(context_lens),
                                   context_lens.shape[0], int(heads_per_read), int(num_ctas),
                                   _ptr(sink), g, ctypes.c_void_p(s.cuda_stream)),
           "pa_kv_read_probe")


def pa_share_groups(block_tables: torch.Tensor, context_lens: torch.Tensor, g: int,
                    mode: int = 1, stream=None):
    """The shared-prefix groups of a batch, as pa_decode's share_prefix=mode
    finds them: (skip [B], groups [B, 3] = (first, members, shared blocks) per
    group then zeros, order [B]); member j of group s is
    order[groups[s, 0] + j]. int32 device tensors."""
    _need_cuda("block_tables", block_tables, torch.int32)
    _need_cuda("context_lens", context_lens, torch.int32)
    B = context_lens.shape[0]
    dev = block_tables.device
    skip = torch.zeros(B, dtype=torch.int32, device=dev)
    groups = torch.zeros(B, 3, dtype=torch.int32, device=dev)
    order = torch.zeros(B, dtype=torch.int32, device=dev)
    s = torch.cuda.current_stream(dev) if stream is None else stream
    _check(_lib().pa_share_groups(_ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B,
                                  int(g), int(mode), _ptr(skip), _ptr(groups), _ptr(order),
                                  ctypes.c_void_p(s.cuda_stream)), "pa_share_groups")
    return skip, groups, order


def pa_decode_default_ctas(k_cache: torch.Tensor, n_h: int, num_seqs: int) -> int:
    r = _lib().pa_decode_default_ctas(geometry(k_cache, n_h), num_seqs)
    if r < 0:
        raise PAError(r, "pa_decode_default_ctas")
    return r


def pa_status_from_device(word: int) -> int:
    return _lib().pa_status_from_device(int(word))


def pa_plan_owner(item: int, total_items: int, num_ctas: int) -> int:
    return _lib().pa_plan_owner(int(item), int(total_items), int(num_ctas))


def pa_version() -> int:
    return _lib().pa_version()


def allocate_pool(num_blocks: int, n_kv: int, d_h: int, kv_dtype: str = "bf16",
                  device="cuda", block_size: int = 16):
    """Zeroed device pool tensors: (k_cache, v_cache, k_scale, v_scale)."""
    shape = (num_blocks, n_kv, block_size, d_h)
    if kv_dtype == "bf16":
        kc = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        vc = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        return kc, vc, None, None
    if kv_dtype in ("int8", "int4"):
        if kv_dtype == "int8":
            kc = torch.zeros(shape, dtype=torch.int8, device=device)
            vc = torch.zeros(shape, dtype=torch.int8, device=device)
        else:
            kc = torch.zeros(shape[:3] + (d_h // 2,), dtype=torch.uint8, device=device)
            vc = torch.zeros(shape[:3] + (d_h // 2,), dtype=torch.uint8, device=device)
        ks = torch.zeros(shape[:3], dtype=torch.float32, device=device)
        vs = torch.zeros(shape[:3], dtype=torch.float32, device=device)
        return kc, vc, ks, vs
    raise ValueError(kv_dtype)


def pa_block_copy(k_cache: torch.Tensor, v_cache: torch.Tensor, pairs: torch.Tensor,
                  k_scale: Optional[torch.Tensor] = None, v_scale: Optional[torch.Tensor] = None,
                  dev_status: Optional[torch.Tensor] = None, stream=None) -> None:
    """Copy pool blocks pairs[p][0] -> pairs[p][1] (int32 [n, 2] on the device),
    K, V and (INT8) scales: the device half of copy-on-write."""
    _need_cuda("k_cache", k_cache)
    _need_cuda("v_cache", v_cache, k_cache.dtype)
    _need_cuda("pairs", pairs, torch.int32)
    if v_cache.shape != k_cache.shape:
        raise ValueError("v_cache must have the shape of k_cache")
    if pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be [num_pairs, 2]")
    g = geometry(k_cache, n_h=k_cache.shape[1])
    if g.kv_dtype != PA_KV_BF16:
        for nm, s in (("k_scale", k_scale), ("v_scale", v_scale)):
            if s is None:
                raise ValueError(f"{nm} is required for an int8/int4 pool")
            _need_cuda(nm, s, torch.float32)
            if tuple(s.shape) != tuple(k_cache.shape[:3]):
                raise ValueError(f"{nm} must be [num_blocks, n_kv, block_size]")
    if dev_status is not None:
        _need_cuda("dev_status", dev_status, torch.int32)
    st = _lib().pa_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(k_scale), _ptr(v_scale),
                              _ptr(pairs), pairs.shape[0], g, _ptr(dev_status),
                              _stream_ptr(stream))
    _check(st, "pa_block_copy")


def _np_ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


def _i32(a, name: str) -> np.ndarray:
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    if a.ndim != 1:
        raise ValueError(f"{name} must be one-dimensional")
    return a


def block_hash(parent: int, token_ids) -> int:
    """One link of the chained block hash (pa_block_hash)."""
    t = _i32(token_ids, "token_ids")
    return int(_lib().pa_block_hash(ctypes.c_uint64(parent), _np_ptr(t), t.shape[0]))


class BlockAllocator:
    """Host block manager of libpa.so (include/pa_alloc.h): reference counts,
    chained-hash prefix caching with an LRU evictable pool, fork, and
    copy-on-write. Block tables are held by the caller as int32 arrays."""

    def __init__(self, num_blocks: int, block_size: int = 16):
        h = ctypes.c_void_p()
        _check(_lib().pa_allocator_create(num_blocks, block_size, ctypes.byref(h)),
               "pa_allocator_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            _lib().pa_allocator_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def allocate_prompt(self, token_ids):
        """-> (block table as an int32 array, cached tokens)."""
        t = _i32(token_ids, "token_ids")
        cap = (t.shape[0] + self.block_size - 1) // self.block_size
        table = np.empty(max(cap, 1), np.int32)
        n, cached = ctypes.c_int32(), ctypes.c_int32()
        _check(_lib().pa_allocator_allocate_prompt(self._h, _np_ptr(t), t.shape[0],
                                                   _np_ptr(table), cap, ctypes.byref(n),
                                                   ctypes.byref(cached)),
               "pa_allocator_allocate_prompt")
        return table[:n.value].copy(), cached.value

    def append_slots(self, tables: np.ndarray, n_blocks: np.ndarray, token_ids):
        """Append one token to each row of `tables` (int32 [B, capacity], updated in
        place with `n_blocks` int32 [B]) -> (slots int64 [B], cow pairs int32 [k, 2]).
        On an error the raised PAError carries .num_done."""
        if tables.dtype != np.int32 or not tables.flags.c_contiguous or tables.ndim != 2:
            raise ValueError("tables must be a C-contiguous int32 [B, capacity] array")
        if n_blocks.dtype != np.int32 or not n_blocks.flags.c_contiguous or \
                n_blocks.shape != (tables.shape[0],):
            raise ValueError("n_blocks must be a C-contiguous int32 [B] array")
        t = _i32(token_ids, "token_ids")
        B = tables.shape[0]
        if t.shape[0] != B:
            raise ValueError("one token id per sequence")
        slots = np.empty(B, np.int64)
        cow = np.empty((max(B, 1), 2), np.int32)
        ncow, ndone = ctypes.c_int32(), ctypes.c_int32()
        st = _lib().pa_allocator_append_slots(self._h, _np_ptr(tables), tables.shape[1],
                                              _np_ptr(n_blocks), _np_ptr(t), B, _np_ptr(slots),
                                              _np_ptr(cow), ctypes.byref(ncow),
                                              ctypes.byref(ndone))
        if st != 0:
            e = PAError(st, "pa_allocator_append_slots")
            e.num_done = ndone.value
            e.cow_pairs = cow[:ncow.value].copy()
            raise e
        return slots, cow[:ncow.value].copy()

    def fork(self, table) -> np.ndarray:
        t = _i32(table, "table")
        _check(_lib().pa_allocator_fork(self._h, _np_ptr(t), t.shape[0]), "pa_allocator_fork")
        return t.copy()

    def free(self, table) -> None:
        t = _i32(table, "table")
        _check(_lib().pa_allocator_free(self._h, _np_ptr(t), t.shape[0]), "pa_allocator_free")

    def num_free(self) -> int:
        return int(_lib().pa_allocator_num_free(self._h))

    def block_info(self, block: int):
        """-> (ref_count, num_tokens, hash or None)."""
        r, n, hh = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        h = ctypes.c_uint64()
        _check(_lib().pa_allocator_block_info(self._h, block, ctypes.byref(r), ctypes.byref(n),
                                              ctypes.byref(h), ctypes.byref(hh)),
               "pa_allocator_block_info")
        return r.value, n.value, (h.value if hh.value else None)

    def free_order(self) -> list:
        out = np.empty(self.num_blocks, np.int32)
        n = ctypes.c_int64()
        _check(_lib().pa_allocator_free_order(self._h, _np_ptr(out), self.num_blocks,
                                              ctypes.byref(n)), "pa_allocator_free_order")
        return out[:n.value].tolist()
