"""pa_kv_read_probe reads exactly the bytes a decode reads: every K/V tile
(and, for INT8/INT4 pools, every scale row) of every block of every
sequence, through the block tables. Its output is an XOR of every 32-bit
word it loaded (folded over CTAs), so it must equal the XOR of the same
multiset of words computed here with numpy, for any CTA count and for one
head or all heads per read."""
import numpy as np
import pytest
import torch

import paged_kv_cache_94_gb300 as pa
from tests.gpu_helpers import gpu_pool
from workloads import Geometry, make_workload

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


def _words(t: torch.Tensor) -> np.ndarray:
    """A device tensor's bytes as uint32 words, per block (first dimension)."""
    a = t.contiguous().view(torch.uint8).cpu().numpy()
    return a.reshape(a.shape[0], -1).view(np.uint32)


def _expected(w, pool) -> int:
    kc, vc, ks, vs = pool
    parts = [_words(kc), _words(vc)] + ([_words(ks), _words(vs)] if ks is not None else [])
    counts = np.zeros(w.num_blocks, np.int64)
    for b in range(w.B):
        counts[w.block_tables[b, :w.num_seq_blocks(b)]] += 1
    odd = np.nonzero(counts % 2)[0]     # a word read twice cancels in the XOR
    x = np.uint32(0)
    for part in parts:
        x ^= np.bitwise_xor.reduce(part[odd].ravel()) if odd.size else np.uint32(0)
    return int(x)


@pytest.mark.parametrize("kv_dtype", ["bf16", "int8", "int4"])
@pytest.mark.parametrize("grid", [1, 7, 304])
def test_read_probe_reads_the_decode_bytes(kv_dtype, grid):
    prefix = [0, 32, 32, 0] if kv_dtype == "int8" else None   # shared blocks read twice
    group = [-1, 0, 0, -1] if kv_dtype == "int8" else None
    ctx = [300, 32 + 70, 32 + 17, 1]
    w = make_workload("probe", Geometry(n_h=8, n_kv=4, d_h=128, kv_dtype=kv_dtype), ctx,
                      seed=8100 + grid, prefix_len=prefix, group=group)
    pool = gpu_pool(w, DEV)
    kc, vc, ks, vs = pool
    want = _expected(w, pool)
    bt = torch.from_numpy(w.block_tables).to(DEV)
    cl = torch.from_numpy(w.context_lens).to(DEV)
    for hg in (1, 2, 4):
        sink = torch.zeros(grid, dtype=torch.int32, device=DEV)
        pa.pa_kv_read_probe(kc, vc, bt, cl, w.geom.n_h, hg, grid, sink, k_scale=ks, v_scale=vs)
        torch.cuda.synchronize()
        got = np.bitwise_xor.reduce(sink.cpu().numpy().view(np.uint32))
        assert int(got) == want, (hg, hex(int(got)), hex(want))
