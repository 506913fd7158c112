#!/usr/bin/env python
"""Benchmark of one paged decode step on GB300.

A step is the whole hot path for one batch: pa_cache_write of every
sequence's new token (slot-mapped append; INT8 quantise for an INT8 pool),
then pa_decode (block-table gather, g-wide q.K, online softmax, P.V, split
merge). Inputs are seeded synthetic tensors resident in HBM before timing.

Metric: KV-read HBM GB/s of the step (algorithmic bytes / time), with the
decode kernel's fraction of the measured HBM peak and sequences/s.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle on the host cores
  python bench.py --op block_copy        # copy-on-write block copies, HBM GB/s
  python bench.py --op allocator         # host block manager, appends/s

With N > 1 (torchrun) every rank runs an independent replica of the same
workload on its own GPU (the path has no cross-GPU exchange): weak scaling,
value = bytes of all ranks / max time over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import CONFIG_NAMES, EXTRA_NAMES, named_workload  # noqa: E402

METRIC = "paged GQA decode attention: KV-read HBM GB/s, % of peak, seqs/s"
DEFAULT_WORKLOAD = "long_context"
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, ~8 TB/s nominal: the gate is 75% of this
L2_FLUSH_BYTES = 512 << 20  # > 129 MB of L2
L2_CLEAN_BYTES = 384 << 20  # read after the write: the L2 then holds clean lines
L2_NOTE = ("flushed between timed steps: a 512 MiB write, then a 384 MiB read so that the "
           "L2 holds clean lines (the write alone leaves ~129 MB of dirty lines whose "
           "write-back would land inside the next timed kernel)")


def max_over_ranks(x: float, world: int, device) -> float:
    """The largest x over all ranks (x itself when world == 1): the timed
    region of a multi-replica run ends when its slowest rank ends."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


class StagedInputs:
    """Tensors packed into one pinned host buffer (each 256-byte aligned) and a
    device buffer of the same layout: one host-to-device copy moves them all."""

    def __init__(self, tensors, dev):
        offs, off = [], 0
        for t in tensors:
            off = (off + 255) // 256 * 256
            offs.append(off)
            off += t.numel() * t.element_size()
        self.nbytes = off
        self.host = torch.empty(off, dtype=torch.uint8).pin_memory()
        self.dev = torch.empty(off, dtype=torch.uint8, device=dev)

        def views(buf):
            return [buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                    for o, t in zip(offs, tensors)]
        for h, t in zip(views(self.host), tensors):
            h.copy_(t.cpu())
        self.device_views = views(self.dev)

    def upload(self):
        self.dev.copy_(self.host, non_blocking=True)


class L2Flush:
    """Evicts the L2 between timed launches, outside the events: writes a
    buffer larger than L2, then reads another one, so the timed kernel starts
    on a cold L2 without the flush's own dirty lines to write back."""

    def __init__(self, dev):
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_CLEAN_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.empty(1, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.sum(self.r, dim=0, keepdim=True, out=self.sink)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", choices=CONFIG_NAMES + EXTRA_NAMES, default=DEFAULT_WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--num-ctas", type=int, default=0, help="force the decode split (tuning)")
    ap.add_argument("--op", choices=["step", "block_copy", "allocator", "read_probe"],
                    default="step",
                    help="step: the decode step (default); block_copy: pa_block_copy; "
                         "allocator: the host block manager; read_probe: plain reads of the "
                         "decode's K/V blocks (the access pattern's ceiling)")
    ap.add_argument("--pairs", type=int, default=4096, help="block pairs per pa_block_copy")
    ap.add_argument("--shuffle", action="store_true",
                    help="decode the batch's sequences in a seeded random order (sharers of a "
                         "prefix are then spread over the batch)")
    ap.add_argument("--no-share", action="store_true",
                    help="decode shared-prefix workloads without the shared-prefix passes")
    return ap.parse_args()


# --------------------------------------------------------------------- bytes
def kv_bits_per_elem(w) -> int:
    return {"bf16": 16, "int8": 8, "int4": 4}[w.geom.kv_dtype]


def scale_bytes_per_row(w) -> int:
    return 0 if w.geom.kv_dtype == "bf16" else 4


def decode_bytes(w, unique_blocks: bool = True) -> dict:
    """Algorithmic bytes of one pa_decode launch.

    Per sequence: ctx*2*n_kv*d_h*b_kv of K and V (+ ctx*2*n_kv*4 of fp32
    scales for INT8), 4*ceil(ctx/16) of block table, 4 of context length, and
    2*2*n_h*d_h of q and out. Shared prefix blocks count once (unique bytes).
    Under a sliding window only the window's tokens and blocks count.
    """
    g = w.geom
    per_token = 2 * g.n_kv * g.d_h * kv_bits_per_elem(w) // 8 + 2 * g.n_kv * scale_bytes_per_row(w)

    def span(b):  # attended positions [lo, ctx) and the blocks they touch
        ctx = int(w.context_lens[b])
        lo = max(0, ctx - w.window) if w.window else 0
        return lo, ctx, range(lo // 16, -(-ctx // 16))

    tok_logical = sum(span(b)[1] - span(b)[0] for b in range(w.B))
    if unique_blocks:
        # attended tokens in unique physical blocks (shared prefixes once)
        seen = set()
        tok = 0
        for b in range(w.B):
            lo, ctx, blocks_b = span(b)
            for i in blocks_b:
                blk = int(w.block_tables[b, i])
                if blk in seen:
                    continue
                seen.add(blk)
                tok += min(16 * i + 16, ctx) - max(16 * i, lo)
    else:
        tok = tok_logical
    blocks = sum(len(span(b)[2]) for b in range(w.B))
    other = 4 * blocks + 4 * w.B + 2 * 2 * w.B * w.n_q * g.n_h * g.d_h
    return {"bytes": tok * per_token + other, "logical_bytes": tok_logical * per_token + other,
            "flops": 4 * g.n_h * g.d_h * tok_logical * w.n_q}


def cache_write_bytes(w) -> int:
    """Bytes of one pa_cache_write of B new tokens: read k, v and slots, write rows."""
    g = w.geom
    rows = w.B * w.n_q * g.n_kv
    read = 2 * rows * g.d_h * 2 + 8 * w.B * w.n_q
    write = 2 * rows * g.d_h * kv_bits_per_elem(w) // 8 + 2 * rows * scale_bytes_per_row(w)
    return read + write


def peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


# Device code of the decode kernel: its DRAM counters depend on these files only.
DECODE_DEVICE_SOURCES = ["pa_ptx.cuh", "pa_plan.h", "pa_internal.h", "pa_decode.cuh",
                         "pa_decode_kernel.cuh", "pa_decode_quant.cuh", "pa_decode_bf16_d128.cu",
                         "pa_decode_bf16_d64.cu", "pa_decode_int8_d128.cu", "pa_decode_int8_d64.cu",
                         "pa_decode_int4_d128.cu", "pa_decode_int4_d64.cu"]


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "paged_kv_cache_94_gb300", "csrc")
    for f in DECODE_DEVICE_SOURCES:
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """ncu DRAM bytes per decode launch, if recorded for the current kernel source."""
    p = os.path.join(ROOT, "profiles", "decode_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p)).get(workload)
    if not d or d.get("kernel_hash") != kernel_source_hash():
        return None
    return d.get("bytes_per_launch")


# -------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        out_dir = os.environ.get("PA_BENCH_OUT", os.path.join(ROOT, "bench_out"))
        self.path = os.path.join(out_dir, f"clocks_rank{index}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


# -------------------------------------------------------------------- oracle
def oracle_sample(w, gen_device, seconds: float):
    """Time the CPU oracle on a bounded sample of the workload's sequences.

    Returns (bytes of the sample, seconds, description). The sample grows one
    sequence at a time until about `seconds` of oracle time is spent.
    """
    import oracle
    from oracle import Pool

    g = w.geom
    done_bytes, spent, seqs = 0, 0.0, []
    order = list(range(w.B))
    q_all = oracle.bf16_bits(w.q(gen_device))
    per_token = 2 * g.n_kv * g.d_h * kv_bits_per_elem(w) // 8 + 2 * g.n_kv * scale_bytes_per_row(w)
    for b in order:
        k, v = w.seq_kv(b, gen_device)
        ctx = int(w.context_lens[b])
        nblk = -(-ctx // 16)
        pool = Pool(nblk, g.n_kv, g.d_h, 16, g.kv_dtype)
        pool.write(oracle.bf16_bits(k), oracle.bf16_bits(v), np.arange(ctx))
        table = np.arange(nblk, dtype=np.int32)[None]
        t0 = time.perf_counter()
        if w.n_q > 1:
            oracle.decode_mq(q_all[b:b + 1], pool, table, np.array([ctx], np.int32), g.n_h,
                             w.scale)
        elif w.window:
            oracle.decode_window(q_all[b:b + 1], pool, table, np.array([ctx], np.int32), g.n_h,
                                 w.scale, window=w.window)
        else:
            oracle.decode(q_all[b:b + 1], pool, table, np.array([ctx], np.int32), g.n_h, w.scale)
        spent += time.perf_counter() - t0
        lo = max(0, ctx - w.window) if w.window else 0
        done_bytes += (ctx - lo) * per_token + 4 * (nblk - lo // 16) + 4 + 4 * w.n_q * g.n_h * g.d_h
        seqs.append(b)
        if spent >= seconds:
            break
    attended = sum(min(int(w.context_lens[s]), w.window) if w.window else int(w.context_lens[s])
                   for s in seqs)
    desc = (f"{len(seqs)} of {w.B} sequences ({attended} attended tokens), "
            f"C fp64 oracle")
    return done_bytes, spent, desc, seqs


def _unit_inputs(w, b, kvh, k, v, q_all):
    """The oracle's inputs for one (sequence, kv head) unit: a compact pool
    holding only that kv head's rows, its g query heads, a 0..n-1 table."""
    import oracle
    from oracle import Pool
    g = w.geom
    ctx = int(w.context_lens[b])
    nblk = -(-ctx // 16)
    pool = Pool(nblk, 1, g.d_h, 16, g.kv_dtype)
    pool.write(oracle.bf16_bits(k[:, kvh:kvh + 1]), oracle.bf16_bits(v[:, kvh:kvh + 1]),
               np.arange(ctx))
    heads = slice(kvh * g.g, (kvh + 1) * g.g)
    q = q_all[b:b + 1, :, heads] if w.n_q > 1 else q_all[b:b + 1, heads]
    return pool, np.ascontiguousarray(q), np.arange(nblk, dtype=np.int32)[None], \
        np.array([ctx], np.int32)


def _oracle_worker(name, units, barrier, commands, results):
    """One host core's share of the all-cores oracle sample. Builds its units'
    pools once (untimed), then for every command waits for all workers and
    times the oracle's decode of its units (wall clock); None ends it."""
    import oracle
    w = named_workload(name)
    g = w.geom
    q_all = oracle.bf16_bits(w.q("cpu"))
    prepared, kv_of = [], {}
    for b, kvh in units:
        if b not in kv_of:
            kv_of.clear()
            kv_of[b] = w.seq_kv(b, "cpu")
        prepared.append(_unit_inputs(w, b, kvh, *kv_of[b], q_all))
    kv_of.clear()
    results.put(None)   # ready
    while commands.get() is not None:
        barrier.wait()
        t0 = time.time()
        for pool, q, table, ctx in prepared:
            if w.n_q > 1:
                oracle.decode_mq(q, pool, table, ctx, g.g, w.scale)
            elif w.window:
                oracle.decode_window(q, pool, table, ctx, g.g, w.scale, window=w.window)
            else:
                oracle.decode(q, pool, table, ctx, g.g, w.scale)
        results.put((t0, time.time()))


class OracleCores:
    """The unmodified oracle on every host core this process may use, over
    the given sequences: their (sequence, kv head) units, which the oracle
    computes independently, dealt in contiguous runs to one spawned process
    per core (spawned: a forked child of a process holding a CUDA context
    can hang). run() times one pass: wall clock from the first start to the
    last end."""

    def __init__(self, w, seqs):
        import multiprocessing as mp
        units = [(b, h) for b in seqs for h in range(w.geom.n_kv)]
        self.cores = max(1, min(len(os.sched_getaffinity(0)), len(units)))
        ctx = mp.get_context("spawn")
        n = self.cores
        barrier, self.results = ctx.Barrier(n), ctx.Queue()
        self.commands = [ctx.Queue() for _ in range(n)]
        self.procs = [ctx.Process(target=_oracle_worker,
                                  args=(w.name, units[i * len(units) // n:(i + 1) * len(units) // n],
                                        barrier, self.commands[i], self.results), daemon=True)
                      for i in range(n)]
        for p in self.procs:
            p.start()
        for _ in self.procs:
            self.results.get()

    def run(self) -> float:
        for c in self.commands:
            c.put(1)
        spans = [self.results.get() for _ in self.procs]
        return max(e for _, e in spans) - min(s for s, _ in spans)

    def close(self):
        for c in self.commands:
            c.put(None)
        for p in self.procs:
            p.join()
            if p.exitcode != 0:
                raise RuntimeError(f"oracle worker exited with {p.exitcode}")


# ------------------------------------------------------------------- native
def run_native(args, rank, world, local_rank):
    import paged_kv_cache_94_gb300 as pa
    from paged_kv_cache_94_gb300 import build as pa_build

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    pa_build.build()
    w = named_workload(args.workload)
    g = w.geom

    # ---- resident inputs: pool with the history, the step's tensors
    kc, vc, ks, vs = pa.allocate_pool(w.num_blocks, g.n_kv, g.d_h, g.kv_dtype, dev)
    for k, v, slots in w.history_chunks(device=dev):
        pa.pa_cache_write(k, v, torch.from_numpy(slots).to(dev), kc, vc, ks, vs)
    q = w.q(dev)
    kn, vn = w.new_kv(dev)
    slots_new = torch.from_numpy(w.new_token_slots()).to(dev)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    if args.shuffle:  # the decode's rows in another order (the cache append is order-free)
        perm = torch.from_numpy(np.random.default_rng(7).permutation(w.B)).to(dev)
        q, bt, cl = q[perm].contiguous(), bt[perm].contiguous(), cl[perm].contiguous()
    out = torch.empty_like(q)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # sequences sharing prefix blocks (prefix caching): attend those blocks once per group
    share = bool((w.group >= 0).any()) and not args.no_share
    share_mode = (2 if args.shuffle else 1) if share else 0  # 2: sharers anywhere in the batch
    ws = pa.decode_workspace(pa.geometry(kc, g.n_h), w.B, dev, args.num_ctas, n_q=w.n_q,
                             share_prefix=share)
    flush = L2Flush(dev)
    torch.cuda.synchronize(dev)

    def attend(q_, bt_, cl_, out_=None, prepare=False):
        o = out if out_ is None else out_
        if w.n_q > 1:  # multi-query step: the n_q new tokens of each sequence at once
            return pa.pa_decode_mq(q_, kc, vc, bt_, cl_, w.scale, out=o, workspace=ws,
                                   dev_status=status, k_scale=ks, v_scale=vs, prepare=prepare)
        return pa.pa_decode(q_, kc, vc, bt_, cl_, w.scale, out=o, k_scale=ks, v_scale=vs,
                            workspace=ws, dev_status=status, num_ctas=args.num_ctas,
                            window=w.window, share_prefix=share_mode, prepare=prepare)

    def step():
        pa.pa_cache_write(kn, vn, slots_new, kc, vc, ks, vs, dev_status=status)
        attend(q, bt, cl)

    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush()
        step()
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)

    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush()  # L2 flush between timed steps (outside the events)
        ev[i][0].record(stream)
        pa.pa_cache_write(kn, vn, slots_new, kc, vc, ks, vs, dev_status=status)
        ev[i][1].record(stream)
        attend(q, bt, cl)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if world > 1:
        torch.distributed.barrier()
    step_ms = [ev[i][0].elapsed_time(ev[i][2]) for i in range(args.steps)]
    write_ms = [ev[i][0].elapsed_time(ev[i][1]) for i in range(args.steps)]
    dec_ms = [ev[i][1].elapsed_time(ev[i][2]) for i in range(args.steps)]
    st = int(status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}: {pa.pa_status_from_device(st)}")

    total_ms = max_over_ranks(sum(step_ms), world, dev)
    ms_per_step = total_ms / args.steps

    db = decode_bytes(w)
    wb = cache_write_bytes(w)
    step_bytes = db["bytes"] + wb
    value = world * step_bytes / (ms_per_step * 1e-3) / 1e9
    dec_avg = statistics.mean(dec_ms)
    pk = peaks()
    achieved = db["bytes"] / (dec_avg * 1e-3) / 1e9

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": g.kv_dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "num_seqs": w.B,
                   "context_tokens": int(w.context_lens.sum()),
                   "l2": L2_NOTE + f"; KV working set {db['bytes'] / 1e6:.0f} MB > 129 MB L2",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "shared_prefix_passes": share, "shuffled": bool(args.shuffle)},
        "seqs_per_s": round(world * w.B / (ms_per_step * 1e-3), 1),
        "decode_ms": round(dec_avg, 5), "cache_write_ms": round(statistics.mean(write_ms), 5),
        "bytes_per_step": step_bytes, "logical_kv_bytes": db["logical_bytes"],
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": recorded_traffic(args.workload),
                     "kernel": ("pa::share_detect_kernel + pa::decode_kernel (shared-prefix "
                                "groups and suffixes in one launch)" if share
                                else "pa::decode_kernel"),
                     "peak_source": pk["source"],
                     "algorithmic_bytes_per_launch": db["bytes"]},
        "gpu_launches": (3 if share else 2) * args.steps,
        "clocks": clocks,
    }

    # ---- end to end through the public API with host buffers
    if not args.no_e2e:
        # Each step's inputs sit in one pinned host buffer (q, new K/V, slots,
        # block tables, context lengths, 256-byte aligned) and move in one
        # copy; its output comes back in one copy. Double-buffered on two copy
        # streams, so step i+1's upload and step i-1's download overlap step
        # i's kernels (a serving loop's pipelining). The KV working set is
        # larger than L2, so this leg runs without flushes; the timed region
        # is the whole loop, copies included.
        hins = [StagedInputs([q, kn, vn, slots_new, bt, cl], dev) for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        houts = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(2)]
        h2d = hins[0].nbytes
        d2h = houts[0].numel() * houts[0].element_size()
        up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        uploaded = [torch.cuda.Event() for _ in range(2)]
        consumed = [torch.cuda.Event() for _ in range(2)]   # step done with inputs and out j
        returned = [torch.cuda.Event() for _ in range(2)]   # out j copied to the host
        for e in uploaded + consumed + returned:
            e.record(stream)
        # the step's two calls, validated once per buffer (pa.Prepared)
        calls = []
        for j in range(2):
            dq, dk, dv, ds, dbt, dcl = hins[j].device_views
            calls.append((pa.pa_cache_write(dk, dv, ds, kc, vc, ks, vs, dev_status=status,
                                            prepare=True),
                          attend(dq, dbt, dcl, outs[j], prepare=True)))

        def e2e_steps(n):
            for i in range(n):
                j = i & 1
                up.wait_event(consumed[j])       # step i-2 is done with buffer j
                with torch.cuda.stream(up):
                    hins[j].upload()
                uploaded[j].record(up)
                stream.wait_event(uploaded[j])
                stream.wait_event(returned[j])   # out j of step i-2 is on the host
                calls[j][0]()                    # pa_cache_write
                calls[j][1]()                    # pa_decode (or pa_decode_mq)
                consumed[j].record(stream)
                down.wait_event(consumed[j])
                with torch.cuda.stream(down):
                    houts[j].copy_(outs[j], non_blocking=True)
                returned[j].record(down)
            stream.wait_stream(up)
            stream.wait_stream(down)

        e2e_steps(args.warmup)
        torch.cuda.synchronize(dev)
        if world > 1:
            torch.distributed.barrier()
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        up.wait_stream(stream)
        e2e_steps(args.steps)
        t1.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(t0.elapsed_time(t1), world, dev) / args.steps
        result["e2e"] = {"value": round(world * step_bytes / (e2e_ms * 1e-3) / 1e9, 2),
                         "unit": "GB/s", "ms_per_step": round(e2e_ms, 5),
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "pipelined": "double-buffered inputs and outputs on two copy streams",
                         "l2": "no flush: the KV working set is larger than L2; no events "
                               "between the step's kernels"}
        result["gpu_launches"] += (3 if share else 2) * args.steps

    # ---- the oracle on the host cores (rank 0 only, N=1 only)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(w, dev, args.cpu_seconds)
    return result


def cpu_baseline(w, dev, seconds):
    """The oracle on the host cores: first one thread on a sample of about
    `seconds`, then every core of the affinity mask on the same sample."""
    nbytes, secs, desc, seqs = oracle_sample(w, dev, seconds)
    pool = OracleCores(w, seqs)
    try:
        wall, cores = pool.run(), pool.cores
    finally:
        pool.close()
    return {"value": round(nbytes / wall / 1e9, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": desc + f", (sequence, kv head) units over {cores} processes",
            "seconds": round(wall, 3),
            "one_thread": {"value": round(nbytes / secs / 1e9, 4), "unit": "GB/s", "cores": 1,
                           "seconds": round(secs, 2)}}


# ---------------------------------------------------------------- read probe
def probe_bytes(w) -> int:
    """Bytes pa_kv_read_probe reads: every block of every sequence, K and V
    (and their scales), and the block-table entries."""
    g = w.geom
    blocks = sum(w.num_seq_blocks(b) for b in range(w.B))
    tile = 16 * g.d_h * kv_bits_per_elem(w) // 8
    scales = 2 * 16 * 4 if g.kv_dtype != "bf16" else 0
    return blocks * g.n_kv * (2 * tile + scales) + 4 * blocks


def run_read_probe(args, rank, world, local_rank):
    """pa_kv_read_probe over the workload's pool: the same scattered blocks as
    its decode, read with plain 16-byte loads, one (block, head) tile at a
    time and all heads of a block at once; L2 flushed between launches."""
    import paged_kv_cache_94_gb300 as pa
    from paged_kv_cache_94_gb300 import build as pa_build

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    pa_build.build()
    w = named_workload(args.workload)
    g = w.geom
    kc, vc, ks, vs = pa.allocate_pool(w.num_blocks, g.n_kv, g.d_h, g.kv_dtype, dev)
    for k, v, slots in w.history_chunks(device=dev):
        pa.pa_cache_write(k, v, torch.from_numpy(slots).to(dev), kc, vc, ks, vs)
    bt = torch.from_numpy(w.block_tables).to(dev)
    cl = torch.from_numpy(w.context_lens).to(dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    grid = args.num_ctas or 4 * sms
    sink = torch.zeros(grid, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    nbytes = probe_bytes(w)
    out = {}
    for hg in sorted({1, g.n_kv}):
        def launch():
            pa.pa_kv_read_probe(kc, vc, bt, cl, g.n_h, hg, grid, sink, k_scale=ks, v_scale=vs)
        for _ in range(args.warmup):
            flush()
            launch()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        for i in range(args.steps):
            flush()
            ev[i][0].record(stream)
            launch()
            ev[i][1].record(stream)
        torch.cuda.synchronize(dev)
        ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
        out[hg] = (ms, nbytes / (ms * 1e-3) / 1e9)
    pk = peaks()
    per_tile, per_block = out[1], out[g.n_kv]
    return {
        "metric": "K/V read probe: HBM GB/s of the decode's scattered reads",
        "value": round(per_tile[1], 2), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(per_tile[0], 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": g.kv_dtype, "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "grid": grid,
                   "l2": L2_NOTE, "reads": "16-byte loads, no arithmetic"},
        "bytes_per_step": nbytes,
        "per_head_tiles": {"ms": round(per_tile[0], 5), "gbs": round(per_tile[1], 1),
                           "frac": round(per_tile[1] / pk["hbm_gbs"], 4)},
        "all_heads_per_block": {"ms": round(per_block[0], 5), "gbs": round(per_block[1], 1),
                                "frac": round(per_block[1] / pk["hbm_gbs"], 4)},
        "peak": pk["hbm_gbs"], "gpu_launches": 2 * args.steps,
    }


# ---------------------------------------------------------------- block copy
def block_copy_bytes(g, pairs: int) -> int:
    """Read + write of every copied block: K and V tiles (+ INT8/INT4 scales)."""
    tile = g.n_kv * 16 * g.d_h * {"bf16": 16, "int8": 8, "int4": 4}[g.kv_dtype] // 8
    scales = 2 * g.n_kv * 16 * 4 if g.kv_dtype != "bf16" else 0
    return 2 * pairs * (2 * tile + scales) + 8 * pairs


def run_block_copy(args, rank, world, local_rank):
    """pa_block_copy of --pairs (source, destination) blocks of the workload's
    pool geometry, one launch per step, L2 flushed between launches."""
    import paged_kv_cache_94_gb300 as pa
    from paged_kv_cache_94_gb300 import build as pa_build
    from workloads import block_copy_pairs

    dev = torch.device(f"cuda:{local_rank}")
    torch.cuda.set_device(dev)
    pa_build.build()
    w = named_workload(args.workload)
    g = w.geom
    nb = max(w.num_blocks, 2 * args.pairs)
    kc, vc, ks, vs = pa.allocate_pool(nb, g.n_kv, g.d_h, g.kv_dtype, dev)
    for t in (kc, vc):
        t.view(torch.uint8).random_(0, 256) if t.dtype != torch.bfloat16 else t.normal_()
    pairs_h = block_copy_pairs(7, nb, args.pairs)
    pairs = torch.from_numpy(pairs_h).to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        flush()
        pa.pa_block_copy(kc, vc, pairs, ks, vs, dev_status=status)
    torch.cuda.synchronize(dev)
    if world > 1:
        torch.distributed.barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    sampler = ClockSampler(local_rank)
    sampler.start()
    time.sleep(0.3)
    for i in range(args.steps):
        flush()
        ev[i][0].record(stream)
        pa.pa_block_copy(kc, vc, pairs, ks, vs, dev_status=status)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    clocks = sampler.stop()
    if int(status.item()) != 0:
        raise RuntimeError(f"device status {int(status.item())}")
    total_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev), world, dev)
    ms = total_ms / args.steps
    nbytes = block_copy_bytes(g, args.pairs)
    achieved = nbytes / (ms * 1e-3) / 1e9
    pk = peaks()
    result = {
        "metric": "copy-on-write block copy: HBM GB/s", "value": round(world * achieved, 2),
        "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": g.kv_dtype,
        "data": "synthetic",
        "config": {"workload": f"pa_block_copy of {args.pairs} blocks, {w.name} pool geometry "
                               f"(n_kv={g.n_kv}, d_h={g.d_h}, {g.kv_dtype})",
                   "l2": L2_NOTE + f"; {nbytes / 2e6:.0f} MB read per launch",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "bytes_per_step": nbytes,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                     "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                     "traffic": None, "kernel": "pa::block_copy_kernel",
                     "peak_source": pk["source"], "algorithmic_bytes_per_launch": nbytes},
        "gpu_launches": args.steps, "clocks": clocks,
    }
    if not args.no_e2e:
        # the copy list comes from the host each step (pinned), as a block manager hands it over
        hp = pairs.cpu().pin_memory()
        dp = torch.empty_like(pairs)
        e2e = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        hst = torch.empty(1, dtype=torch.int32).pin_memory()
        for i in range(args.steps):
            flush()
            e2e[i][0].record(stream)
            dp.copy_(hp, non_blocking=True)
            pa.pa_block_copy(kc, vc, dp, ks, vs, dev_status=status)
            hst.copy_(status, non_blocking=True)
            e2e[i][1].record(stream)
        torch.cuda.synchronize(dev)
        e_ms = sum(a.elapsed_time(b) for a, b in e2e) / args.steps
        result["e2e"] = {"value": round(world * nbytes / (e_ms * 1e-3) / 1e9, 2), "unit": "GB/s",
                         "ms_per_step": round(e_ms, 5), "h2d_bytes_per_step": hp.numel() * 4,
                         "d2h_bytes_per_step": 4}
        result["gpu_launches"] += args.steps
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        from oracle.allocator import block_copy as oracle_copy
        def host(t):
            return t.view(torch.int16).cpu().numpy() if t.dtype == torch.bfloat16 else t.cpu().numpy()
        k_h, v_h = host(kc), host(vc)
        ks_h = ks.cpu().numpy() if ks is not None else None
        vs_h = vs.cpu().numpy() if vs is not None else None
        n, spent = 0, 0.0
        while spent < min(args.cpu_seconds, 5.0) and n < args.pairs:
            t0 = time.perf_counter()
            oracle_copy(k_h, v_h, pairs_h[n:n + 256].tolist(), ks_h, vs_h)
            spent += time.perf_counter() - t0
            n = min(args.pairs, n + 256)
        result["cpu_baseline"] = {"value": round(block_copy_bytes(g, n) / spent / 1e9, 3),
                                  "unit": "GB/s", "cores": 1, "kind": "oracle",
                                  "sample": f"{n} of {args.pairs} pairs, numpy block copy"}
    return result


# ----------------------------------------------------------------- allocator
def allocator_trace(seed: int, num_seqs: int, prompt_len: int, shared: int, steps: int):
    """A serving trace for the block manager: num_seqs prompts whose first
    `shared` tokens are common (prefix-cache hits), four-way parallel
    sampling of each, then `steps` decode steps of one token per branch."""
    rng = np.random.default_rng(seed)
    common = rng.integers(0, 32000, shared).tolist()
    prompts = [common + rng.integers(0, 32000, prompt_len - shared).tolist()
               for _ in range(num_seqs)]
    tokens = rng.integers(0, 32000, (steps, 4 * num_seqs)).astype(np.int32)
    return prompts, tokens


def run_allocator(args):
    """Host block manager: appends/s over a serving trace (prefill with prefix
    hits, fork, decode steps with copy-on-write), native vs the oracle."""
    import paged_kv_cache_94_gb300 as pa
    from paged_kv_cache_94_gb300 import build as pa_build
    pa_build.build()
    B, P, S, T = 64, 1000, 512, 256
    cap = (P + T) // 16 + 2
    prompts, tokens = allocator_trace(5, B, P, S, T)
    nblocks = 4 * B * cap

    def native_once():
        a = pa.BlockAllocator(nblocks)
        tables = np.zeros((4 * B, cap), np.int32)
        nb = np.zeros(4 * B, np.int32)
        for i, p in enumerate(prompts):
            t, _ = a.allocate_prompt(p)
            for j in range(4):
                row = a.fork(t) if j else t
                tables[4 * i + j, :len(row)] = row
                nb[4 * i + j] = len(row)
        t0 = time.perf_counter()
        for s in range(T):
            a.append_slots(tables, nb, tokens[s])
        return time.perf_counter() - t0

    def oracle_once(steps):
        from oracle.allocator import Allocator
        a = Allocator(nblocks)
        tabs = []
        for p in prompts:
            t, _ = a.allocate_for_prompt(p)
            tabs += [t] + [a.fork(t) for _ in range(3)]
        t0 = time.perf_counter()
        for s in range(steps):
            for i, t in enumerate(tabs):
                a.append_slot(t, int(tokens[s, i]))
        return time.perf_counter() - t0

    for _ in range(max(1, args.warmup)):
        native_once()
    reps = max(1, min(args.steps, 20))
    secs = [native_once() for _ in range(reps)]
    per = statistics.median(secs)
    appends = 4 * B * T
    o_steps = 32
    o_secs = oracle_once(o_steps)
    return {
        "metric": "block manager: appended tokens/s (decode step with copy-on-write)",
        "value": round(appends / per, 1), "unit": "tokens/s", "n_gpus": 0, "steps": reps,
        "warmup": max(1, args.warmup), "ms_per_step": round(1e3 * per / T, 5),
        "higher_is_better": True, "scaling": "none", "vs_baseline": None, "dtype": "int32",
        "data": "synthetic",
        "config": {"workload": f"{B} prompts of {P} tokens sharing a {S}-token prefix, "
                               f"4 sampled branches each, {T} decode steps of {4 * B} appends",
                   "ms_per_step": "per decode step of the batch (one append_slots call)"},
        "gpu_launches": 0,
        "cpu_baseline": {"value": round(4 * B * o_steps / o_secs, 1), "unit": "tokens/s",
                         "cores": 1, "kind": "oracle",
                         "sample": f"{o_steps} of {T} decode steps, Python oracle allocator"},
    }


# ---------------------------------------------------------------- reference
def run_reference(args):
    """The CPU oracle as the reference arm: each step is the oracle on a
    bounded sample of the workload, on the host cores."""
    w = named_workload(args.workload)
    # the sample: the sequences one thread covers in a few seconds, run on
    # every host core at each step
    nbytes, _, desc, seqs = oracle_sample(w, "cpu", 3.0)
    pool = OracleCores(w, seqs)
    cores = pool.cores
    try:
        for _ in range(args.warmup):
            pool.run()
        tot_b, tot_s = 0, 0.0
        for _ in range(args.steps):
            tot_s += pool.run()
            tot_b += nbytes
    finally:
        pool.close()
    value = tot_b / tot_s / 1e9
    g = w.geom
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot_s / args.steps, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{w.name}: {w.description}", "num_seqs": w.B},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle",
                         "sample": desc + f" per step, (sequence, kv head) units over {cores} "
                                          "processes"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return
    if args.op == "allocator":
        if rank == 0:
            print(json.dumps(run_allocator(args)), flush=True)
        return
    if world > 1:
        torch.distributed.init_process_group(
            backend="nccl", device_id=torch.device(f"cuda:{local_rank}"))
    try:
        if args.op == "block_copy":
            res = run_block_copy(args, rank, world, local_rank)
        elif args.op == "read_probe":
            res = run_read_probe(args, rank, world, local_rank)
        else:
            res = run_native(args, rank, world, local_rank)
        if rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
