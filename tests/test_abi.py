"""Host-side checks of the C ABI (no GPU needed, no compute calls).

The library must load and export every entry point include/*.h declares;
argument checks that return before any CUDA call are exercised; the work
split (pa_plan_owner) is compared with a brute-force assignment.
"""
import ctypes
import os
import re

import pytest

import paged_kv_cache_94_gb300 as pa
from paged_kv_cache_94_gb300 import build as pa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    pa_build.build()
    return pa.library()


def _declared():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if f.endswith(".h"):
            text = re.sub(r"/\*.*?\*/", "", open(os.path.join(inc, f)).read(), flags=re.S)
            names |= set(re.findall(r"\b(pa_[a-z_0-9]+)\s*\(", text))
    return sorted(names)


def test_header_declares_the_binding_names():
    assert sorted(pa.EXPORTED) == _declared()


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name
        getattr(lib, name)


def test_status_strings_and_device_words(lib):
    for code, name in pa.STATUS.items():
        assert lib.pa_status_string(code).decode().startswith(name)
    assert lib.pa_status_from_device(0) == 0
    assert lib.pa_status_from_device(pa.PA_DEV_BAD_BLOCK | pa.PA_DEV_BAD_SLOT) == -5
    assert lib.pa_status_from_device(pa.PA_DEV_BAD_SLOT) == -6
    assert lib.pa_status_from_device(pa.PA_DEV_BAD_CONTEXT) == -9
    assert lib.pa_status_from_device(pa.PA_DEV_TIMEOUT) == -10
    assert lib.pa_version() >= 100


def _geom(**kw):
    base = dict(num_blocks=100, n_h=32, n_kv=8, d_h=128, block_size=16, kv_dtype=0, reserved=0)
    base.update(kw)
    return pa.pa_geom(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(n_h=30), -2),           # n_h % n_kv != 0
    (dict(n_kv=0), -2),
    (dict(num_blocks=0), -2),
    (dict(kv_dtype=7), -3),
    (dict(d_h=96), -4),
    (dict(block_size=32), -4),
    (dict(n_h=24, n_kv=1), -4),   # group 24 not compiled
    (dict(reserved=1), -2),
    (dict(num_blocks=1 << 27), -4),  # TMA row coordinate overflow
])
def test_cache_write_rejects_bad_geometry_before_launch(lib, kw, status):
    fake = ctypes.c_void_p(256)  # never dereferenced: the call returns before any launch
    st = lib.pa_cache_write(fake, fake, fake, 4, fake, fake, None, None, _geom(**kw), None, None)
    assert st == status


def test_cache_write_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    g = _geom()
    assert lib.pa_cache_write(fake, fake, fake, 0, fake, fake, None, None, g, None, None) == 0
    assert lib.pa_cache_write(fake, fake, fake, -1, fake, fake, None, None, g, None, None) == -2
    assert lib.pa_cache_write(None, fake, fake, 4, fake, fake, None, None, g, None, None) == -1
    # bf16 pools take no scales; int8 pools need them
    assert lib.pa_cache_write(fake, fake, fake, 4, fake, fake, fake, fake, g, None, None) == -2
    g8 = _geom(kv_dtype=1)
    assert lib.pa_cache_write(fake, fake, fake, 4, fake, fake, None, None, g8, None, None) == -1
    odd = ctypes.c_void_p(258)
    assert lib.pa_cache_write(odd, fake, fake, 4, fake, fake, None, None, g, None, None) == -11


def test_decode_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    g = _geom()
    args = lambda **o: [o.get("q", fake), fake, fake, o.get("ks"), o.get("vs"), fake,
                        o.get("mb", 16), fake, o.get("B", 4), 0.1, fake, o.get("ws", fake),
                        1 << 20, o.get("g", g), None, None]
    assert lib.pa_decode(*args(B=0)) == 0          # nothing to do
    assert lib.pa_decode(*args(B=-1)) == -2
    assert lib.pa_decode(*args(B=9000)) == -2
    assert lib.pa_decode(*args(mb=0)) == -2
    assert lib.pa_decode(*args(q=None)) == -1
    assert lib.pa_decode(*args(ws=None)) == -7
    assert lib.pa_decode(*args(ks=fake, vs=fake)) == -2
    assert lib.pa_decode(*args(g=_geom(kv_dtype=1))) == -1
    assert lib.pa_decode(*args(q=ctypes.c_void_p(264))) == -11
    assert lib.pa_decode(*args(ws=ctypes.c_void_p(272))) == -11
    assert lib.pa_decode_ex(*args(), 0) == -2
    mq = args()[:9] + [2] + args()[9:]   # n_q = 2 after num_seqs
    assert lib.pa_decode_mq_ex(*mq, 0) == -2    # num_ctas must be > 0
    mq[9] = 0
    assert lib.pa_decode_mq_ex(*mq, 8) == -2    # n_q must be >= 1
    assert lib.pa_decode_workspace_size(_geom(n_h=30), 4, 0) == 0


def test_plan_owner_matches_brute_force(lib):
    for W, grid in [(1, 1), (8, 12), (13, 4), (100, 7), (65536, 304), (163840, 152), (999, 1000)]:
        G = min(grid, W)  # never more CTAs than items
        lo = [c * W // G for c in range(G + 1)]
        owner = [None] * W
        for c in range(G):
            for x in range(lo[c], lo[c + 1]):
                owner[x] = c
        step = max(1, W // 2000)
        for x in list(range(0, W, step)) + [W - 1]:
            assert lib.pa_plan_owner(x, W, grid) == owner[x], (W, grid, x)
        # every CTA's range is non-empty and within one item of W/G, so the
        # owners of a run of items are a run of CTAs with no gaps
        sizes = [lo[c + 1] - lo[c] for c in range(G)]
        assert min(sizes) >= 1 and max(sizes) - min(sizes) <= 1
    assert lib.pa_plan_owner(5, 5, 3) == -1
    # lines whose W * G passes 2^32 take 64-bit arithmetic, the others 32-bit:
    # the owner of x is the c with floor(c W / G) <= x < floor((c+1) W / G)
    import random
    rng = random.Random(5)
    for W, grid in [(2**32 // 456, 456), (2**32 // 456 + 1, 456), (10**9, 1000), (3 * 10**9, 8000)]:
        G = min(grid, W)
        for x in [0, 1, W - 2, W - 1] + [rng.randrange(W) for _ in range(200)]:
            c = lib.pa_plan_owner(x, W, grid)
            assert c * W // G <= x < (c + 1) * W // G, (W, grid, x, c)


def test_binding_refuses_cpu_tensors():
    import torch
    q = torch.zeros(1, 4, 64, dtype=torch.bfloat16)
    kc = torch.zeros(2, 2, 16, 64, dtype=torch.bfloat16)
    bt = torch.zeros(1, 1, dtype=torch.int32)
    cl = torch.ones(1, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA"):
        pa.pa_decode(q, kc, kc, bt, cl, 0.125)


def test_block_copy_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    odd = ctypes.c_void_p(258)
    g = _geom()
    assert lib.pa_block_copy(fake, fake, None, None, fake, 0, g, None, None) == 0  # nothing to do
    assert lib.pa_block_copy(fake, fake, None, None, fake, -1, g, None, None) == -2
    assert lib.pa_block_copy(None, fake, None, None, fake, 3, g, None, None) == -1
    assert lib.pa_block_copy(fake, fake, None, None, None, 3, g, None, None) == -1
    assert lib.pa_block_copy(fake, fake, fake, None, fake, 3, g, None, None) == -2  # bf16 + scales
    gi = _geom(kv_dtype=1)
    assert lib.pa_block_copy(fake, fake, None, None, fake, 3, gi, None, None) == -1
    assert lib.pa_block_copy(odd, fake, None, None, fake, 3, g, None, None) == -11
    assert lib.pa_block_copy(fake, fake, None, None, fake, 3, _geom(d_h=96), None, None) == -4


def test_decode_opt_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    dec = [fake, fake, fake, None, None, fake, 4, fake, 2, ctypes.c_float(0.1), fake, fake,
           ctypes.c_size_t(1 << 20)]

    def call(g, **kw):
        o = pa.pa_decode_opts(**{**dict(window=0, n_sink=0, sink_k=None, sink_v=None,
                                        num_ctas=0, share_prefix=0, reserved=0), **kw})
        return lib.pa_decode_opt(*dec, g, ctypes.byref(o), None, None)

    g = _geom()
    assert call(g, window=-1) == -2
    assert call(g, reserved=3) == -2
    assert call(g, n_sink=4, sink_k=256, sink_v=256) == -2          # sink rows need INT8
    gi = _geom(kv_dtype=1)
    assert call(gi, n_sink=17, sink_k=256, sink_v=256) == -2
    assert call(gi, n_sink=4, sink_k=None, sink_v=256) == -1
    assert call(gi, n_sink=4, sink_k=257, sink_v=256) == -11
    assert call(g, share_prefix=3) == -2 and call(g, share_prefix=-1) == -2
    assert call(g, share_prefix=2) != -2                            # sharers anywhere: valid
    assert call(g, share_prefix=1, window=64) == -4                 # not with a window
    assert call(_geom(n_h=128, n_kv=8), share_prefix=1) == -4      # g = 16


@pytest.mark.parametrize("kv_dtype", [0, 1, 2])
def test_mq_workspace_size_per_pool_type(lib, kv_dtype):
    # multi-query kernels exist for every pool type at g * n_q <= 16 (explicit
    # CTA count: no device query); other shapes report 0
    for n_h, n_q, ok in [(16, 2, True), (16, 8, True), (32, 4, True), (64, 2, True),
                         (32, 8, False), (16, 3, False), (128, 2, False)]:
        g = _geom(n_h=n_h, n_kv=8, kv_dtype=kv_dtype)
        size = lib.pa_decode_mq_workspace_size(g, 4, n_q, 304)
        assert (size > 0) == ok, (n_h, n_q, kv_dtype)


def test_read_probe_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    g = _geom()
    args = lambda **o: [fake, fake, None, None, fake, 16, fake, o.get("B", 4),
                        o.get("hg", 1), o.get("grid", 8), fake, o.get("g", g), None]
    assert lib.pa_kv_read_probe(*args(B=0)) == 0          # nothing to read
    assert lib.pa_kv_read_probe(*args(hg=3)) == -2        # must divide n_kv
    assert lib.pa_kv_read_probe(*args(hg=0)) == -2
    assert lib.pa_kv_read_probe(*args(grid=0)) == -2
    assert lib.pa_kv_read_probe(*args(g=_geom(kv_dtype=1))) == -2   # INT8 pools read scales
    assert lib.pa_kv_read_probe(*args(g=_geom(d_h=96))) == -2


def test_share_groups_argument_checks(lib):
    fake = ctypes.c_void_p(256)
    call = lambda B=4, mb=16, g=1, mode=1, bt=fake, cl=fake, out=fake: lib.pa_share_groups(
        bt, mb, cl, B, g, mode, out, out, out, None)
    assert call(B=0) == 0                      # nothing to do
    assert call(B=-1) == -2 and call(B=8193) == -2 and call(mb=0) == -2
    assert call(mode=0) == -2 and call(mode=3) == -2
    assert call(g=3) == -4 and call(g=16) == -4
    assert call(bt=None) == -1 and call(out=None) == -1
