"""Seeded synthetic inputs for paged decode attention.

This module builds INPUTS only: query rows, per-token K/V rows, context lengths,
block tables and the slot of every token a caller would append. It holds none of
the attention, softmax or quantisation arithmetic: both the CUDA library and the
CPU oracle receive what this module produces and do their own work on it.

Shapes follow the layer geometries the source pages use:
  * "LLM 推理底层：KV Cache 显存几何、GQA/MLA 压缩与 PagedAttention 调度"
    (blog.faulkner.fun), section "KV Cache 容量公式": Llama-3-70B with
    n_h=64, n_kv=8, d_h=128, B=16, S=8192.
  * "【infra之路】10-PagedAttention 与 KV Cache 管理" (qwbw.cn), §2.1 and §5:
    LLaMA-7B with 32 KV heads, head_dim 128 and block_size 16.
  * "kv-cache-guide" (guijiagi.com), §2.3 table: LLaMA-2/3 layer shapes.

Block tables are a seeded random permutation of the physical pool dealt out in
sequence order, so consecutive logical blocks land on scattered physical blocks,
as the block-table figure of qwbw.cn §3.3 shows.

Token rows are generated per "stream" with a generator seeded from
(workload seed, stream id), so any one sequence's K/V history can be rebuilt on
its own without generating the whole pool. A stream is either one sequence's
private tokens or one group's shared prefix.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Iterator, Optional

import numpy as np
import torch

BLOCK_SIZE = 16

# Value profiles of q, K and V. "normal" draws every element from N(0, 1);
# the others reshape those draws to reach the dynamic range real K/V has:
#   rising       keys climb a staircase along the context (RISE_LEVELS steps
#                of RISE_PERIOD tokens, about RISE_NATS of score each, then
#                back down); queries lean along the same direction
#   v_range      V rows scaled per (token, kv head) by 10**U(-3, 3)
#   kv_range     K and V rows both scaled that way, independently
#   q_big, q_small, q_zero   queries times 1e3, times 1e-3, or zero
#   same_keys    one key row per kv head shared by every position
#   onehot       keys e_(j mod d_h); each sequence's first new token has key
#                2 * e_ONEHOT_DIM and every query is e_ONEHOT_DIM
#   sink_outlier position 0 of each sequence has a key about SINK_NATS above
#                the typical score (the outlier first token that motivates
#                keeping sink tokens, "kv-cache-guide" §4.3)
PROFILES = ("normal", "rising", "v_range", "kv_range", "q_big", "q_small", "q_zero",
            "same_keys", "onehot", "sink_outlier")
RISE_PERIOD = 48
RISE_LEVELS = 12
RISE_NATS = 8.0
SINK_NATS = 12.5
ONEHOT_DIM = 5


@dataclass(frozen=True)
class Geometry:
    """Per-layer attention geometry: query heads, KV heads, head dim, KV dtype."""

    n_h: int
    n_kv: int
    d_h: int
    block_size: int = BLOCK_SIZE
    kv_dtype: str = "bf16"  # "bf16" or "int8"

    @property
    def g(self) -> int:
        return self.n_h // self.n_kv


@dataclass
class Workload:
    """One decode step's worth of paged-attention inputs.

    context_lens[b] counts every token of sequence b INCLUDING the new token,
    which sits at position context_lens[b]-1 and is appended by the step itself.
    Positions 0..context_lens[b]-2 are history that is written into the pool
    before the step (``history_chunks``).
    """

    name: str
    geom: Geometry
    seed: int
    context_lens: np.ndarray          # int32 [B]
    block_tables: np.ndarray          # int32 [B, max_blocks]; unused entries = -1
    num_blocks: int
    scale: float
    prefix_len: np.ndarray            # int32 [B]: shared-prefix tokens of each seq (0 = none)
    group: np.ndarray                 # int32 [B]: shared-prefix group id (-1 = none)
    description: str = ""
    window: int = 0                   # > 0: the step attends the last `window` tokens only
    n_q: int = 1                      # new tokens per sequence (> 1: multi-query step)
    profile: str = "normal"           # value distribution of q, K and V (see PROFILES)
    # streams are generated lazily; cache of (stream id) -> (k, v) on a device
    _cache: dict = field(default_factory=dict, repr=False)

    # ------------------------------------------------------------------ sizes
    @property
    def B(self) -> int:
        return int(self.context_lens.shape[0])

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.B else 0

    def num_seq_blocks(self, b: int) -> int:
        return -(-int(self.context_lens[b]) // self.geom.block_size)

    # ---------------------------------------------------------------- streams
    def _stream_seed(self, stream: int) -> int:
        return (self.seed * 1_000_003 + 7919 * (stream + 1)) & 0x7FFF_FFFF_FFFF

    def _gen_rows(self, stream: int, n: int, device, pos0: int = 0
                  ) -> tuple[torch.Tensor, torch.Tensor]:
        """K and V rows of `n` consecutive positions of one stream, starting at
        sequence position pos0: bf16 [n, n_kv, d_h]."""
        gen = torch.Generator(device=device)
        gen.manual_seed(self._stream_seed(stream))
        shape = (n, self.geom.n_kv, self.geom.d_h)
        k = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        v = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        if self.profile != "normal":
            k, v = self._shape_rows(k, v, gen, stream, pos0, device)
        return k.to(torch.bfloat16), v.to(torch.bfloat16)

    def _direction(self, device) -> torch.Tensor:
        """A fixed +-1 vector per kv head, float32 [n_kv, d_h]: the direction
        the "rising" and "sink_outlier" profiles add to q and to keys."""
        gen = torch.Generator(device=device)
        gen.manual_seed(self._stream_seed(3_000_000))
        bits = torch.randint(0, 2, (self.geom.n_kv, self.geom.d_h), generator=gen, device=device)
        return bits.to(torch.float32) * 2 - 1

    def _shape_rows(self, k, v, gen, stream, pos0, device):
        """Apply the workload's value profile to freshly drawn N(0,1) rows."""
        n, n_kv, d = k.shape
        pos = torch.arange(pos0, pos0 + n, device=device)
        prof = self.profile
        if prof == "rising":
            # a staircase along the context, RISE_LEVELS steps of RISE_PERIOD
            # tokens, then back to the bottom: each step adds about RISE_NATS
            # to every score of a query leaning along the direction
            level = ((pos // RISE_PERIOD) % RISE_LEVELS).to(torch.float32)
            step = RISE_NATS / math.sqrt(d)
            k = k + (level * step)[:, None, None] * self._direction(device)[None]
        elif prof in ("v_range", "kv_range"):
            # per (token, kv head) magnitudes log-uniform over 1e-3 .. 1e3
            amp_v = 10.0 ** (torch.rand((n, n_kv, 1), generator=gen, device=device) * 6 - 3)
            v = v * amp_v
            if prof == "kv_range":
                amp_k = 10.0 ** (torch.rand((n, n_kv, 1), generator=gen, device=device) * 6 - 3)
                k = k * amp_k
        elif prof == "same_keys":
            # every key of every sequence equals one fixed row per kv head
            g2 = torch.Generator(device=device)
            g2.manual_seed(self._stream_seed(3_000_001))
            row = torch.randn((1, n_kv, d), generator=g2, device=device)
            k = row.expand(n, n_kv, d).clone()
        elif prof == "onehot":
            # key at position j is the unit vector e_(j mod d_h); in a
            # sequence's private rows, the row of its first new token is
            # 2 * e_ONEHOT_DIM instead, the only key with a score of 2 * scale
            k = torch.zeros_like(k)
            k[torch.arange(n, device=device), :, pos % d] = 1.0
            if stream < 1_000_000 and n - self.n_q >= 0:
                j = n - self.n_q
                k[j] = 0.0
                k[j, :, ONEHOT_DIM] = 2.0
        elif prof == "sink_outlier":
            # position 0 of every sequence carries a key leaning along the
            # direction, about SINK_NATS above the typical score
            if pos0 == 0 and n > 0:
                k[0] = k[0] + (SINK_NATS / math.sqrt(d)) * self._direction(device)
        elif prof not in ("q_big", "q_small", "q_zero"):
            raise ValueError(f"unknown profile {prof}")
        return k, v

    def _prefix_stream(self, grp: int) -> int:
        return 1_000_000 + grp

    def seq_kv(self, b: int, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
        """K and V rows of every position of sequence b: bf16 [ctx_b, n_kv, d_h]."""
        ctx = int(self.context_lens[b])
        p = int(self.prefix_len[b])
        ks, vs = [], []
        if p > 0:
            kp, vp = self._gen_rows(self._prefix_stream(int(self.group[b])), p, device)
            ks.append(kp)
            vs.append(vp)
        ko, vo = self._gen_rows(b, ctx - p, device, pos0=p)
        ks.append(ko)
        vs.append(vo)
        return torch.cat(ks, 0), torch.cat(vs, 0)

    def q(self, device="cpu") -> torch.Tensor:
        """Query rows of the step: bf16 [B, n_h, d_h], or [B, n_q, n_h, d_h]
        for a multi-query step."""
        gen = torch.Generator(device=device)
        gen.manual_seed(self._stream_seed(2_000_000))
        shape = (self.B, self.geom.n_h, self.geom.d_h)
        if self.n_q > 1:
            shape = (self.B, self.n_q) + shape[1:]
        x = torch.randn(shape, generator=gen, device=device)
        prof = self.profile
        if prof in ("rising", "sink_outlier"):
            # every query head leans along its kv head's direction (the
            # noise halved so that <u, q> stays near d_h for every head)
            u = self._direction(device).repeat_interleave(self.geom.g, dim=0)
            x = 0.5 * x + u
        elif prof == "q_big":
            x = x * 1e3
        elif prof == "q_small":
            x = x * 1e-3
        elif prof == "q_zero":
            x = torch.zeros_like(x)
        elif prof == "onehot":
            x = torch.zeros_like(x)
            x[..., ONEHOT_DIM] = 1.0
        return x.to(torch.bfloat16)

    # ------------------------------------------------------------------ slots
    def slot_of(self, b: int, pos: np.ndarray) -> np.ndarray:
        """Slot a block manager hands out for position(s) pos of sequence b.

        This is the caller-side input of the cache append (the block manager
        owns the table; it tells the kernel where each new row goes).
        """
        bs = self.geom.block_size
        pos = np.asarray(pos, dtype=np.int64)
        return self.block_tables[b, pos // bs].astype(np.int64) * bs + pos % bs

    def new_token_slots(self) -> np.ndarray:
        """int64 [B * n_q]: slots of each sequence's new tokens (positions
        ctx-n_q .. ctx-1, sequence-major); -1 for a position < 0 (a padding row
        the append skips)."""
        out = []
        for b in range(self.B):
            ctx = int(self.context_lens[b])
            for pos in range(ctx - self.n_q, ctx):
                out.append(self.slot_of(b, np.array([pos]))[0] if pos >= 0 else -1)
        return np.array(out, dtype=np.int64)

    def new_kv(self, device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
        """K/V rows of the new tokens of every sequence: bf16 [B * n_q, n_kv, d_h]
        (zeros where the position is < 0)."""
        ks, vs = [], []
        z = torch.zeros((self.geom.n_kv, self.geom.d_h), dtype=torch.bfloat16, device=device)
        for b in range(self.B):
            ctx = int(self.context_lens[b])
            p = int(self.prefix_len[b])
            ko = vo = None
            if ctx > 0:
                assert max(ctx - self.n_q, 0) >= p, "new tokens must be private to their sequence"
                ko, vo = self._gen_rows(b, ctx - p, device, pos0=p)
            for pos in range(ctx - self.n_q, ctx):
                ks.append(ko[pos - p] if pos >= 0 else z)
                vs.append(vo[pos - p] if pos >= 0 else z)
        return torch.stack(ks), torch.stack(vs)

    def history_chunks(self, device="cpu", max_rows: int = 1 << 20,
                       seqs: Optional[list[int]] = None
                       ) -> Iterator[tuple[torch.Tensor, torch.Tensor, np.ndarray]]:
        """Yield (k, v, slots) covering every history position exactly once.

        History = positions 0..ctx-1-n_q of each sequence. A shared prefix is
        yielded once, by the first sequence of its group. ``seqs`` restricts the
        output to those sequences (their shared prefix included).
        """
        done_groups = set()
        order = range(self.B) if seqs is None else seqs
        for b in order:
            ctx = int(self.context_lens[b])
            p = int(self.prefix_len[b])
            grp = int(self.group[b])
            if p > 0 and grp not in done_groups:
                done_groups.add(grp)
                k, v = self._gen_rows(self._prefix_stream(grp), p, device)
                yield from self._chunk(k, v, self.slot_of(b, np.arange(p)), max_rows)
            n_priv = ctx - self.n_q - p
            if n_priv > 0:
                k, v = self._gen_rows(b, ctx - p, device, pos0=p)
                yield from self._chunk(k[:n_priv], v[:n_priv],
                                       self.slot_of(b, np.arange(p, ctx - self.n_q)), max_rows)

    @staticmethod
    def _chunk(k, v, slots, max_rows):
        for s in range(0, k.shape[0], max_rows):
            yield k[s:s + max_rows], v[s:s + max_rows], slots[s:s + max_rows]

    # ------------------------------------------------------------- accounting
    def unique_blocks(self) -> int:
        """Distinct physical blocks referenced by the block tables."""
        ids = set()
        for b in range(self.B):
            ids.update(self.block_tables[b, :self.num_seq_blocks(b)].tolist())
        return len(ids)

    def logical_blocks(self) -> int:
        return sum(self.num_seq_blocks(b) for b in range(self.B))


# ---------------------------------------------------------------------------
# builders
# ---------------------------------------------------------------------------

def _deal_tables(rng_perm: np.ndarray, context_lens: np.ndarray, block_size: int,
                 prefix_len: np.ndarray, group: np.ndarray, max_blocks: int) -> np.ndarray:
    """Hand out physical IDs from a shuffled pool in sequence order.

    Sequences of one prefix group reuse the group's prefix block IDs.
    """
    B = context_lens.shape[0]
    tables = np.full((B, max_blocks), -1, dtype=np.int32)
    nxt = 0
    group_prefix: dict[int, np.ndarray] = {}
    for b in range(B):
        nblk = -(-int(context_lens[b]) // block_size)
        pblk = int(prefix_len[b]) // block_size
        col = 0
        if pblk > 0:
            grp = int(group[b])
            if grp not in group_prefix:
                group_prefix[grp] = rng_perm[nxt:nxt + pblk].copy()
                nxt += pblk
            tables[b, :pblk] = group_prefix[grp]
            col = pblk
        n = nblk - col
        tables[b, col:nblk] = rng_perm[nxt:nxt + n]
        nxt += n
    assert nxt <= rng_perm.shape[0], "pool too small"
    return tables


def make_workload(name: str, geom: Geometry, context_lens, seed: int,
                  pool_factor: float = 1.1, num_blocks: Optional[int] = None,
                  prefix_len=None, group=None, scale: Optional[float] = None,
                  extra_table_cols: int = 0, description: str = "",
                  window: int = 0, n_q: int = 1, profile: str = "normal") -> Workload:
    """Build a workload from explicit context lengths.

    pool_factor: the physical pool holds ceil(pool_factor * blocks needed) blocks
    (unless num_blocks is given), so some blocks stay unused.
    """
    ctx = np.asarray(context_lens, dtype=np.int32)
    B = ctx.shape[0]
    bs = geom.block_size
    pl = np.zeros(B, np.int32) if prefix_len is None else np.asarray(prefix_len, np.int32)
    gr = np.full(B, -1, np.int32) if group is None else np.asarray(group, np.int32)
    # a shared prefix is whole blocks (the blocks a group's members point at)
    assert (pl % bs == 0).all(), "prefix_len must be a multiple of the block size"
    nblk = [-(-int(c) // bs) for c in ctx]
    # blocks actually handed out (a shared prefix counts once per group)
    needed = 0
    seen = set()
    for b in range(B):
        pblk = int(pl[b]) // bs
        if pblk and int(gr[b]) not in seen:
            seen.add(int(gr[b]))
            needed += pblk
        needed += nblk[b] - pblk
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * needed))
    assert num_blocks >= needed
    gen = torch.Generator().manual_seed(seed)
    perm = torch.randperm(num_blocks, generator=gen).numpy().astype(np.int32)
    max_blocks = max(nblk) + extra_table_cols if B else 1
    tables = _deal_tables(perm, ctx, bs, pl, gr, max(max_blocks, 1))
    if scale is None:
        scale = 1.0 / math.sqrt(geom.d_h)
    if profile not in PROFILES:
        raise ValueError(f"unknown profile {profile}")
    return Workload(name=name, geom=geom, seed=seed, context_lens=ctx, block_tables=tables,
                    num_blocks=int(num_blocks), scale=float(scale), prefix_len=pl, group=gr,
                    description=description, window=int(window), n_q=int(n_q),
                    profile=profile)


# ---------------------------------------------------------------------------
# the five named workloads
# ---------------------------------------------------------------------------

CONFIG_NAMES = ["tiny", "llama3_8b", "llama3_70b", "llama2_7b_int8_prefix", "long_context"]
# further workloads of the variants built beside the decode step
EXTRA_NAMES = ["mistral_7b_window", "llama3_8b_int4", "llama3_8b_spec4"]


def named_workload(name: str) -> Workload:
    """The named workloads, seeded with 94 + their index in CONFIG_NAMES + EXTRA_NAMES."""
    idx = (CONFIG_NAMES + EXTRA_NAMES).index(name)
    seed = 94 + idx
    if name == "tiny":
        return make_workload(
            name, Geometry(n_h=4, n_kv=2, d_h=64), [5, 37], seed, num_blocks=8,
            description="B=2, ctx {5,37}, n_h=4, n_kv=2, d_h=64, pool of 8 blocks")
    if name == "llama3_8b":
        rng = np.random.default_rng(seed)
        ctx = rng.integers(512, 4096, size=64, endpoint=True)
        return make_workload(
            name, Geometry(n_h=32, n_kv=8, d_h=128), ctx, seed,
            description="Llama-3-8B layer: B=64, ctx U[512,4096], n_h=32, n_kv=8, d_h=128, bf16")
    if name == "llama3_70b":
        return make_workload(
            name, Geometry(n_h=64, n_kv=8, d_h=128), [8192] * 16, seed,
            description="Llama-3-70B layer: B=16, ctx 8192, n_h=64, n_kv=8, d_h=128, bf16")
    if name == "llama2_7b_int8_prefix":
        rng = np.random.default_rng(seed)
        suffix = np.clip(np.round(rng.lognormal(mean=6.0, sigma=1.0, size=32)), 16, 4096).astype(np.int64)
        prefix = 2048
        ctx = prefix + suffix
        grp = np.repeat(np.arange(4), 8)
        return make_workload(
            name, Geometry(n_h=32, n_kv=32, d_h=128, kv_dtype="int8"), ctx, seed,
            prefix_len=np.full(32, prefix), group=grp,
            description="LLaMA-2-7B MHA layer, INT8 KV: B=32 in 4 groups of 8 sharing a "
                        "2048-token prefix, suffix lognormal(6,1) clipped to [16,4096]")
    if name == "mistral_7b_window":
        # "kv-cache-guide" (guijiagi.com) §5.2: window w = 4096 over sequences
        # of up to s = 32768 tokens; Mistral-7B layer shape (GQA 32/8, d 128)
        rng = np.random.default_rng(seed)
        ctx = rng.integers(16384, 32768, size=16, endpoint=True)
        return make_workload(
            name, Geometry(n_h=32, n_kv=8, d_h=128), ctx, seed, window=4096,
            description="Mistral-7B layer, sliding window 4096: B=16, ctx U[16384,32768], "
                        "n_h=32, n_kv=8, d_h=128, bf16")
    if name == "llama3_8b_int4":
        # the Llama-3-8B step with an INT4 cache ("kv-cache-guide" §4.2, num_bits 4)
        rng = np.random.default_rng(seed)
        ctx = rng.integers(512, 4096, size=64, endpoint=True)
        return make_workload(
            name, Geometry(n_h=32, n_kv=8, d_h=128, kv_dtype="int4"), ctx, seed,
            description="Llama-3-8B layer, INT4 KV: B=64, ctx U[512,4096], n_h=32, n_kv=8, "
                        "d_h=128")
    if name == "llama3_8b_spec4":
        # speculative verification ("LLM 推理引擎设计" §6): the Llama-3-8B batch
        # checks a 4-token draft per sequence in one multi-query step
        rng = np.random.default_rng(seed)
        ctx = rng.integers(512, 4096, size=64, endpoint=True)
        return make_workload(
            name, Geometry(n_h=32, n_kv=8, d_h=128), ctx, seed, n_q=4,
            description="Llama-3-8B layer, 4-token speculative verify: B=64, ctx U[512,4096], "
                        "n_q=4, n_h=32, n_kv=8, d_h=128, bf16")
    if name == "long_context":
        return make_workload(
            name, Geometry(n_h=32, n_kv=8, d_h=128), [131072, 98304, 65536, 32768], seed,
            description="long context: B=4, ctx {131072,98304,65536,32768}, n_h=32, n_kv=8, d_h=128")
    raise KeyError(name)


# ------------------------------------------------------------ free-form inputs
def random_rows(seed: int, n: int, n_kv: int, d_h: int) -> tuple[torch.Tensor, torch.Tensor]:
    """Seeded K and V rows, bf16 [n, n_kv, d_h] on the CPU (standard normal)."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    k = torch.randn((n, n_kv, d_h), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    v = torch.randn((n, n_kv, d_h), generator=gen, dtype=torch.float32).to(torch.bfloat16)
    return k, v


def random_queries(seed: int, B: int, n_h: int, d_h: int) -> torch.Tensor:
    """Seeded query rows, bf16 [B, n_h, d_h] on the CPU (standard normal)."""
    gen = torch.Generator()
    gen.manual_seed(seed)
    return torch.randn((B, n_h, d_h), generator=gen, dtype=torch.float32).to(torch.bfloat16)


def block_copy_pairs(seed: int, num_blocks: int, n: int) -> np.ndarray:
    """n (source, destination) block pairs: distinct destinations, none of
    them a source, drawn from a seeded permutation of the pool. int32 [n, 2]."""
    assert 2 * n <= num_blocks
    perm = np.random.default_rng(seed).permutation(num_blocks).astype(np.int32)
    return np.ascontiguousarray(np.stack([perm[:n], perm[n:2 * n]], axis=1))
