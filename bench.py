#!/usr/bin/env python
"""Benchmark of one mixed continuous-batching step of paged attention.

One step = the whole hot path on one batch: slot mapping, the cache write of
every new token, and attention of every query row (split-KV decode + combine
for decode rows, tensor-core prefill for chunk rows), through the C ABI.

Default workload (one layer, Llama-3-8B shapes: 32 q / 8 kv heads, d=128,
bf16, block size 16): a 512-token prefill chunk over 1536 cached tokens,
8 fresh 64-token prefills and 1280 decodes with contexts uniform in
[128, 2048] -- 2304 new tokens, about 5.7 GB of K/V read per step, so the
inputs are far larger than L2 and no flush is needed.

Prints one JSON line (rank 0). ``--impl reference`` times the CPU oracle on
a bounded per-step sample of the same workload instead.
"""

import os

# Each oracle process runs numpy single-threaded (one process per host core),
# so that the core count it reports is exact.
for _v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import argparse  # noqa: E402
import hashlib  # noqa: E402
import json  # noqa: E402
import re  # noqa: E402
import subprocess  # noqa: E402
import sys  # noqa: E402
import time  # noqa: E402

import numpy as np  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_hkv_gb300 import synth  # noqa: E402

METRIC = "mixed-step attention tokens/s per layer"
DEFAULT_SEEDS = {"mixed_step": 3, "prefill_rows": 3, "mixed_step_2048": 3, "tiny_decode": 1,
                 "llama_decode": 2, "prefix_sharing": 4, "long_context": 5, "long_prefill": 6}
UNIT = "tokens/s"


def parse_args():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--workload", default="mixed_step", choices=sorted(synth.WORKLOADS))
    p.add_argument("--seed", type=int, default=None)
    p.add_argument("--block-size", type=int, default=16, choices=[8, 16, 32],
                   help="tokens per cache block")
    p.add_argument("--graph", action="store_true",
                   help="time the step as a CUDA graph captured once and replayed")
    p.add_argument("--shared-prefix", choices=["auto", "off"], default="auto",
                   help="pass the shared-prefix hint when the workload's sharing requests "
                        "form one run of decodes (auto), or never (off)")
    p.add_argument("--write", choices=["separate", "fused", "attention"], default="attention",
                   help="slot mapping and cache write as two launches (separate), fused into "
                        "one (pkv_slot_mapping_and_write), or inside the attention call's "
                        "first launch (pkv_paged_attention_with_write)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    return p.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# ------------------------------------------------------------------ ranks
def replica_seed(base_seed, rank):
    """Each rank runs its own replica of the workload with its own batch."""
    return base_seed + rank


def max_over_ranks(value, dist=None, device="cpu"):
    """The slowest rank's time (every rank must call it)."""
    if dist is None:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, max_ms_per_step):
    """Units all ranks processed per second, over the slowest rank's time."""
    return units_per_rank * world / (max_ms_per_step * 1e-3)


# ------------------------------------------------------------------ work
L2_BYTES = 129 * 2 ** 20  # GB300 L2
HBM_NOMINAL_GBS = 7900.0  # GB300 HBM3e, nominal


def step_work(step):
    """Algorithmic bytes and flops of one step.

    decode_kv_bytes: the K and V rows the decode rows read, each physical
    block once (a block shared by several requests counts the most tokens
    any of them keeps in it; Hkv * D * 2 bytes per row); that is the least
    the decode must bring from memory. decode_kv_logical_bytes: the same
    per request (L * Hkv * D * 2 * 2 each), shared blocks once per reader.
    prefill_flops: 4 * D * Hq per causal (query, key) pair (QK^T and PV);
    write_bytes: each new token's K and V rows read and written."""
    D, Hq, Hkv = step.head_dim, step.num_q_heads, step.num_kv_heads
    dec = step.query_len == 1
    row = Hkv * D * 2 * 2
    decode_logical = int(step.seq_lens[dec].astype(np.int64).sum()) * row
    B = step.block_size
    fill = {}
    for r in np.flatnonzero(dec):
        L = int(step.seq_lens[r])
        for j in range(-(-L // B)):
            blk = int(step.block_table[r, j])
            fill[blk] = max(fill.get(blk, 0), min(B, L - j * B))
    decode_kv = sum(fill.values()) * row
    pairs = 0
    for c, n in zip(step.num_computed[~dec], step.query_len[~dec]):
        c, n = int(c), int(n)
        pairs += n * c + n * (n + 1) // 2
    return {
        "decode_kv_bytes": decode_kv,
        "decode_kv_logical_bytes": decode_logical,
        # bytes a step touches at least once: the K/V of every allocated block
        # slot (a shared prefix once), q and out rows
        "touched_bytes": (block_tradeoff(step)["slots_allocated"] * Hkv * D * 2 * 2
                          + 2 * step.num_tokens * Hq * D * 2),
        "decode_rows": int(dec.sum()),
        "prefill_pairs": pairs,
        "prefill_flops": 4 * D * Hq * pairs,
        "write_bytes": 2 * step.num_tokens * Hkv * D * 2 * 2,
        "tokens": step.num_tokens,
    }


def block_tradeoff(step):
    """The block-size trade-off of one step's cache: slots allocated but
    holding no token (internal fragmentation of last blocks) and the block
    table entries the attention reads.

    Blocks shared by several requests count once; a block's stored tokens
    are the most any request keeps in it."""
    B = step.block_size
    fill = {}
    entries = 0
    for r in range(step.num_reqs):
        L = int(step.seq_lens[r])
        n = -(-L // B)
        entries += n
        for j in range(n):
            blk = int(step.block_table[r, j])
            fill[blk] = max(fill.get(blk, 0), min(B, L - j * B))
    allocated = len(fill) * B
    stored = sum(fill.values())
    return {"table_entries_read": entries, "blocks_in_use": len(fill),
            "slots_allocated": allocated,
            "slots_wasted_frac": (allocated - stored) / allocated if allocated else 0.0}


def kernels_per_step(step, fused_write=False, shared_prefix=None, write_in_attention=False):
    """Launches of one step: slot mapping and write (one launch when fused,
    none of their own inside the attention call), the plan, the prefill
    (prefill rows or shared-prefix items), decode and combine."""
    write = 0 if write_in_attention else (1 if fused_write else 2)
    return write + 1 + (1 if step.max_query_len > 1 or shared_prefix else 0) + 2


# ------------------------------------------------------------------ clocks
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.sel = []
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(device_index).uuid)
            self.sel = ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            self.sel = []

    def start(self):
        cmd = ["nvidia-smi"] + self.sel + [f"--query-gpu={self.FIELDS}",
                                           "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.06)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for n, v in zip(names, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "samples": len(sm), "reasons": sorted(reasons)}


REJECT_REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown")


def clocks_rejected(clocks):
    """A timed region whose clock samples show a hardware or thermal
    slowdown, or an SM clock held well below its maximum with no reason given
    (a clock lock left by someone else), is not a valid measurement.
    sw_power_cap alone is kept (and reported)."""
    if any(r in REJECT_REASONS for r in clocks.get("reasons", [])):
        return True
    sm, smax = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and smax and sm < 0.9 * smax and not clocks.get("reasons"))


# ------------------------------------------------------------------ oracle timing
# Rows of one step the CPU oracle computes per class of request, at most: the
# mixed step (1280 decodes, one 512-row chunk, 8 x 64 prefill rows) fits in
# full; larger workloads are sampled.
ORACLE_ROW_CAP = {"decode": 1280, "chunk": 512, "prefill": 512}
ORACLE_CLASSES = ("decode", "chunk", "prefill")


def request_class(spec):
    if spec.query_len == 1:
        return "decode"
    return "chunk" if spec.num_computed > 0 else "prefill"


def oracle_plan(step_specs, seed, caps, workers):
    """Rows the oracle computes, split over the host workers.

    For each class of request (decodes, chunks over a cached prefix, fresh
    prefills) every row is taken when the class has at most ``caps[class]``
    rows, else a seeded sample of that many. Rows go round-robin to the
    workers; a worker builds every request it holds rows of. Returns
    {class: (per-worker [(request index, row in request)], total rows of
    the class, rows taken)}."""
    rng = np.random.default_rng(seed + 1000)
    plan = {}
    for key in ORACLE_CLASSES:
        pairs = [(i, j) for i, sp in enumerate(step_specs) if request_class(sp) == key
                 for j in range(sp.query_len)]
        if not pairs:
            continue
        take = pairs
        if len(pairs) > caps[key]:
            idx = np.sort(rng.choice(len(pairs), size=caps[key], replace=False))
            take = [pairs[k] for k in idx]
        per = [take[w::workers] for w in range(workers)]
        plan[key] = (per, len(pairs), len(take))
    return plan


def _oracle_worker(conn):
    """One host process of the oracle timing. It builds its share of the
    requests when told to ("build"), then runs the oracle on them each time
    it is told to ("run"); the parent times each run over all workers."""
    import oracle
    built = {}
    while True:
        msg = conn.recv()
        if msg is None:
            conn.close()
            return
        op, arg = msg
        if op == "build":
            built = {}
            for key, specs, rows, shape, seed in arg:
                reqs = sorted({i for i, _ in rows})
                if not reqs:
                    continue
                pos = {i: k for k, i in enumerate(reqs)}
                sub = synth.make_step([specs[i] for i in reqs], seed=seed, **shape)
                sel = [int(sub.query_start_loc[pos[i]]) + j for i, j in rows]
                built[key] = (sub, sel)
            conn.send("ready")
        elif op == "run":
            item = built.get(arg)
            if item is not None:
                sub, sel = item
                slots = oracle.slot_mapping(sub.block_table, sub.query_start_loc,
                                            sub.num_computed, sub.block_size)
                pool = oracle.kv_write(sub.kv_cache, sub.k, sub.v, slots)
                oracle.paged_attention(sub.q, pool, sub.block_table, sub.seq_lens,
                                       sub.query_start_loc, sub.num_computed, sub.scale,
                                       rows=sel)
            conn.send("done")


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover - non-Linux hosts
        return os.cpu_count() or 1


class OracleTimer:
    """The CPU oracle on every host core: one spawned process per core
    (numpy single-threaded in each), fed one step's rows by oracle_plan.
    ``time_step`` runs the step's classes one after another, each as one
    wall-clock region over all workers, and scales each class to its full
    row count."""

    def __init__(self, step_specs, shape, seed, caps=ORACLE_ROW_CAP, workers=None):
        import multiprocessing as mp
        self.workers = workers or host_cores()
        self.plan = oracle_plan(step_specs, seed, caps, self.workers)
        ctx = mp.get_context("spawn")  # no fork after CUDA is up
        self.conns, self.procs = [], []
        for _ in range(self.workers):
            a, b = ctx.Pipe()
            proc = ctx.Process(target=_oracle_worker, args=(b,), daemon=True)
            proc.start()
            self.conns.append(a)
            self.procs.append(proc)
        for w, conn in enumerate(self.conns):
            conn.send(("build", [(key, step_specs, per[w], shape, seed)
                                 for key, (per, _, _) in self.plan.items()]))
        for conn in self.conns:
            if conn.recv() != "ready":
                raise RuntimeError("oracle worker failed to build its inputs")

    def _run(self, key):
        t0 = time.perf_counter()
        for conn in self.conns:
            conn.send(("run", key))
        for conn in self.conns:
            if conn.recv() != "done":
                raise RuntimeError("oracle worker failed")
        return time.perf_counter() - t0

    def time_step(self):
        """(estimated seconds for the whole step, seconds actually timed)."""
        est = timed = 0.0
        for key, (_, total, taken) in self.plan.items():
            dt = self._run(key)
            timed += dt
            est += dt * total / taken
        return est, timed

    @property
    def full_step(self):
        return all(total == taken for _, total, taken in self.plan.values())

    def describe(self):
        parts = []
        for key, (_, total, taken) in self.plan.items():
            parts.append(f"{key}: {taken} of {total} rows" if taken < total
                         else f"{key}: all {total} rows")
        return (f"{'the whole step' if self.full_step else 'a seeded sample of the step'} "
                f"({'; '.join(parts)}) on {self.workers} processes, one per host core")

    def close(self):
        for conn in self.conns:
            try:
                conn.send(None)
            except (BrokenPipeError, OSError):
                pass
        for proc in self.procs:
            proc.join(timeout=10)


def shape_of(step):
    return dict(num_q_heads=step.num_q_heads, num_kv_heads=step.num_kv_heads,
                head_dim=step.head_dim, block_size=step.block_size)


# ------------------------------------------------------------------ reference arm
def run_reference(args):
    """The CPU oracle as the reference arm: every step is the workload's
    step (the whole mixed step; larger workloads sampled per class, see
    ORACLE_ROW_CAP) computed by the oracle on all host cores."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    seed = args.seed if args.seed is not None else DEFAULT_SEEDS[args.workload]
    meta = synth.WORKLOADS[args.workload](seed=seed, materialize=False,
                                          block_size=args.block_size)
    timer = OracleTimer(meta.specs, shape_of(meta), seed)
    try:
        for _ in range(args.warmup):
            timer.time_step()
        est, timed = [], []
        for _ in range(args.steps):
            e, t = timer.time_step()
            est.append(e)
            timed.append(t)
    finally:
        timer.close()
    sec = float(np.mean(est))
    value = meta.num_tokens / sec
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3,
        # the step time is measured when every row of the step runs; for a
        # sampled workload it is the per-class extrapolation of the timed rows
        "ms_per_step_is_estimate": not timer.full_step,
        "sample_ms_per_step_timed": float(np.mean(timed)) * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": args.workload, "tokens_per_step": meta.num_tokens,
                   "block_size": args.block_size},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": timer.workers, "kind": "oracle",
                         "sample": "per step: " + timer.describe()},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))
    return 0


# ------------------------------------------------------------------ native arm
def code_sha256(text):
    """sha256 of a C/CUDA source's code with comments, indentation and empty
    lines removed, so that editing a comment does not count as changing the
    kernel. (The sources put no comment markers inside string literals.)"""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    lines = [ln.strip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def traffic_from_profile(kernel_src):
    """DRAM traffic per launch of the decode kernel from the committed ncu
    figures (profiles/decode_traffic.json), if they were taken on the
    current code (else None)."""
    path = os.path.join(ROOT, "profiles", "decode_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    with open(kernel_src, encoding="utf-8") as f:
        if code_sha256(f.read()) != rec.get("code_sha256"):
            return None
    return float(rec["traffic_bytes_per_launch"])


def run_e2e(ds, step, work, K, world, pg, sync_all):
    """The step end to end through the public calls, as a serving loop runs
    it: every step uploads all of its inputs (q, k, v, block table, lengths)
    from pinned host memory and downloads its whole output. The inputs sit
    back to back in one pinned staging buffer, so each step's upload is one
    copy. Two sets of device buffers alternate between steps, and the uploads
    and downloads run on their own streams, so step k+1's upload and step
    k-1's download overlap step k's kernels. The cache pool is shared (the
    steps run in order on one stream)."""
    import torch

    from paged_kv_cache_hkv_gb300.runner import DeviceStep

    ds2 = DeviceStep(step, upload_pool=False, shared_prefix=ds.shared_prefix,
                     fused_write=ds.fused_write, write_in_attention=ds.write_in_attention)
    ds2.kv_cache = ds.kv_cache
    sets = [ds, ds2]
    names = ("q", "k", "v", "block_table", "seq_lens", "query_start_loc", "num_computed")
    # one staging layout: each input at a 256-byte aligned offset
    offs, total = [], 0
    for n in names:
        t = getattr(ds, n)
        offs.append(total)
        total += -(-(t.numel() * t.element_size()) // 256) * 256
    host_stage = torch.empty(total, dtype=torch.uint8, pin_memory=True)
    for n, o in zip(names, offs):
        t = getattr(ds, n)
        nb = t.numel() * t.element_size()
        host_stage[o:o + nb].copy_(t.reshape(-1).view(torch.uint8).cpu())
    dev_stage = []
    for cur in sets:  # the set's input tensors become views of one device buffer
        buf = torch.empty(total, dtype=torch.uint8, device="cuda")
        for n, o in zip(names, offs):
            t = getattr(cur, n)
            nb = t.numel() * t.element_size()
            setattr(cur, n, buf[o:o + nb].view(t.dtype).view(t.shape))
        dev_stage.append(buf)
    host_out = [torch.empty(ds.out.shape, dtype=ds.out.dtype, pin_memory=True) for _ in sets]
    h2d = total
    d2h = host_out[0].numel() * host_out[0].element_size()
    compute = torch.cuda.current_stream()
    up, down = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    uploaded, computed, downloaded = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    sync_all()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(compute)
    up.wait_event(e0)
    down.wait_event(e0)
    for k in range(K):
        b = k % 2
        cur = sets[b]
        with torch.cuda.stream(up):  # inputs of step k, once step k-2 is done with the set
            if k >= 2:
                up.wait_event(computed[b])
            dev_stage[b].copy_(host_stage, non_blocking=True)
            uploaded[b].record(up)
        compute.wait_event(uploaded[b])
        if k >= 2:  # the set's previous output has left the device
            compute.wait_event(downloaded[b])
        cur.run(stream=compute)
        computed[b].record(compute)
        with torch.cuda.stream(down):
            down.wait_event(computed[b])
            host_out[b].copy_(cur.out, non_blocking=True)
            downloaded[b].record(down)
    compute.wait_stream(up)
    compute.wait_stream(down)
    e1.record(compute)
    sync_all()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), pg, device="cuda")
    # every step computes the same batch: the last download must equal the
    # device-resident result
    if not torch.equal(host_out[(K - 1) % 2], ds.out.cpu()):
        raise SystemExit("end-to-end output differs from the device-resident step")
    return {"value": whole_job_rate(work["tokens"], world, e2e_ms / K), "unit": UNIT,
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "overlap": "one staged upload and one download per step, on their own streams, "
                       "two buffer sets"}


def timed_region(ds, run_step, K, stream, device_index, sync_all):
    """K timed steps (CUDA events on the launching stream, clocks sampled
    meanwhile), then a separate run of min(K, 100) steps with events recorded
    between the kernels for per-kernel times. Returns the K steps' total ms,
    the median ms per launch of (plan, prefill, decode, combine), the cache
    write's median ms per launch and the clock summary."""
    import torch

    from paged_kv_cache_hkv_gb300 import binding

    t_start, t_stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device_index)
    sync_all()
    sampler.start()
    time.sleep(0.15)
    sync_all()
    t_start.record(stream)
    for _ in range(K):
        run_step()
    t_stop.record(stream)
    sync_all()
    # per-kernel times from a separate run with events recorded between the
    # kernels of the attention call
    KT = min(K, 100)
    trace = [[torch.cuda.Event(enable_timing=True) for _ in range(binding.PKV_TRACE_EVENTS)]
             for _ in range(KT)]
    write_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(KT)]
    for ev in trace:  # torch creates the CUDA event on its first record
        for e in ev:
            e.record(stream)
    for a, b in write_ev:
        a.record(stream)
        b.record(stream)
    sync_all()
    s = ds.step
    for k in range(KT):
        ds.slot_map()
        write_ev[k][0].record(stream)
        ds.write()
        write_ev[k][1].record(stream)
        binding.pkv_paged_attention(
            ds.out, ds.q, ds.kv_cache, ds.block_table, ds.seq_lens, ds.query_start_loc,
            ds.num_computed, max_query_len=s.max_query_len, max_seq_len=s.max_seq_len,
            scale=s.scale, workspace=ds.workspace, trace_events=trace[k],
            shared_prefix=ds.shared_prefix)
    sync_all()
    # the cache write alone, back to back (each launch rewrites the same rows,
    # so every one moves the full bytes): its time per launch without the
    # launch latency that a single bracketed launch carries
    NW = 50
    w0, w1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    calls = ds.calls()
    run_step()  # the GPU works on a step while the writes are queued behind it
    w0.record(stream)
    for _ in range(NW):
        calls.write()
    w1.record(stream)
    # the same rows through the slot mapping fused into the write (the per-token
    # routine that the one-call step runs inside its first launch)
    m0, m1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    run_step()
    m0.record(stream)
    for _ in range(NW):
        calls.slot_map_and_write()
    m1.record(stream)
    sync_all()
    write_b2b_ms = w0.elapsed_time(w1) / NW
    mapped_b2b_ms = m0.elapsed_time(m1) / NW
    clocks = sampler.stop()
    total_ms = t_start.elapsed_time(t_stop)
    # ms per launch, the median over the traced steps: plan, prefill, decode, combine
    per_kernel = np.median(np.array([[ev[i].elapsed_time(ev[i + 1])
                                      for i in range(binding.PKV_TRACE_EVENTS - 1)]
                                     for ev in trace]), axis=0)
    write_ms = (float(np.median([a.elapsed_time(b) for a, b in write_ev])), write_b2b_ms,
                mapped_b2b_ms)
    return total_ms, per_kernel, write_ms, clocks


def run_native(args):
    import torch

    from paged_kv_cache_hkv_gb300 import binding
    from paged_kv_cache_hkv_gb300.runner import DeviceStep

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py: no CUDA device (the native arm has no CPU path)")
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist

    base_seed = args.seed if args.seed is not None else DEFAULT_SEEDS[args.workload]
    seed = replica_seed(base_seed, rank)
    step = synth.WORKLOADS[args.workload](seed=seed, block_size=args.block_size)
    ds = DeviceStep(step, shared_prefix="auto" if args.shared_prefix == "auto" else None,
                    fused_write=args.write == "fused",
                    write_in_attention=args.write == "attention")
    binding.pkv_get_device_errors(clear=True)
    work = step_work(step)
    stream = torch.cuda.current_stream()

    def sync_all():
        torch.cuda.synchronize()
        if pg is not None:
            pg.barrier()

    for _ in range(max(args.warmup, 3)):
        ds.run()
    torch.cuda.synchronize()
    flags = binding.pkv_get_device_errors(clear=True)
    if flags:
        raise SystemExit(f"device error flags {flags:#x} during warm-up")

    K = args.steps
    # the step as a user runs it: nothing between the kernels, so each one may
    # start its prologue while the one before finishes (or, with --graph, the
    # three calls captured once into a CUDA graph and replayed)
    run_step = ds.run
    if args.graph:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            ds.run()
        stream.wait_stream(side)
        graph.replay()
        run_step = graph.replay
        sync_all()
    total_ms, per_kernel, write_ms, clocks = timed_region(ds, run_step, K, stream, local, sync_all)
    # taken again once (and that one reported) if any rank's clocks were off;
    # every rank decides the same, so their barriers stay matched
    if max_over_ranks(1.0 if clocks_rejected(clocks) else 0.0, pg, device="cuda") > 0:
        first = clocks
        total_ms, per_kernel, write_ms, clocks = timed_region(ds, run_step, K, stream, local,
                                                              sync_all)
        clocks["remeasured_after"] = first["reasons"] or [f"sm {first['sm_mhz']} MHz"]
    total_ms = max_over_ranks(total_ms, pg, device="cuda")
    ms_per_step = total_ms / K
    value = whole_job_rate(work["tokens"], world, ms_per_step)
    flags = binding.pkv_get_device_errors(clear=True)
    if flags:
        raise SystemExit(f"device error flags {flags:#x} in the timed region")

    # ---- end to end: host inputs in, host output out, every step
    e2e = None
    if not args.no_e2e:
        e2e = run_e2e(ds, step, work, K, world, pg, sync_all)

    # ---- roofline of the dominant kernel (decode)
    peaks = {}
    try:
        peaks = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
        hbm_peak, peak_src = float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        hbm_peak, peak_src = 6800.0, "fallback"
    dec_ms = per_kernel[2]
    dec_gbs = work["decode_kv_bytes"] / (dec_ms * 1e-3) / 1e9 if dec_ms > 0 else None
    # the committed counters cover the default mixed step only
    traffic = None
    if args.workload == "mixed_step" and args.block_size == 16 and args.seed is None:
        traffic = traffic_from_profile(os.path.join(ROOT, "paged_kv_cache_hkv_gb300", "csrc",
                                                    "decode.cu"))
    # The measured peak is a read+write copy; a read-only stream (the decode)
    # runs a few percent above it, so frac can exceed 1. The chip's nominal
    # HBM3e bandwidth is given beside it as an upper reference.
    roofline = {"kernel": "decode_kernel", "bound": "hbm", "achieved": dec_gbs,
                "peak": hbm_peak, "peak_source": peak_src, "unit": "GB/s",
                "frac": dec_gbs / hbm_peak if dec_gbs else None, "traffic": traffic,
                "algorithmic_bytes_per_launch": work["decode_kv_bytes"],
                "peak_nominal": HBM_NOMINAL_GBS,
                "frac_of_nominal": dec_gbs / HBM_NOMINAL_GBS if dec_gbs else None}
    pf_ms = per_kernel[1]
    tc_peak = float(peaks.get("bf16_tflops", 1900.0))
    prefill = None
    if work["prefill_flops"] and pf_ms > 0:
        tf = work["prefill_flops"] / (pf_ms * 1e-3) / 1e12
        # the burst peak: the launches here run for at most milliseconds (the
        # seconds-long sustained figure is given beside it for context)
        tc_sus = float(peaks.get("bf16_tflops_sustained", 0.0)) or None
        prefill = {"kernel": "prefill_kernel", "bound": "tensor", "achieved": tf,
                   "peak": tc_peak, "unit": "TFLOP/s", "frac": tf / tc_peak,
                   "peak_sustained": tc_sus, "frac_of_sustained": tf / tc_sus if tc_sus else None,
                   "algorithmic_flops_per_launch": work["prefill_flops"]}

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        timer = OracleTimer(step.specs, shape_of(step), seed)
        try:
            sec, timed = timer.time_step()
        finally:
            timer.close()
        cpu = {"value": work["tokens"] / sec, "unit": UNIT, "cores": timer.workers,
               "kind": "oracle", "sample": timer.describe(),
               "seconds_timed": timed, "extrapolated": not timer.full_step}

    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "tokens_per_step": work["tokens"],
                   "requests": step.num_reqs, "decode_rows": work["decode_rows"],
                   "heads": f"{step.num_q_heads}q/{step.num_kv_heads}kv", "head_dim": step.head_dim,
                   "block_size": step.block_size, "pool_blocks": step.num_blocks,
                   "decode_kv_bytes_per_step": work["decode_kv_bytes"],
                   "decode_kv_logical_bytes_per_step": work["decode_kv_logical_bytes"],
                   "prefill_flops_per_step": work["prefill_flops"],
                   "l2": ("inputs larger than L2 (no flush)" if work["touched_bytes"] > L2_BYTES
                          else "inputs fit in L2 (no flush: L2-warm timings)"),
                   "shared_prefix_hint": (dict(zip(("len", "first_req", "num_reqs"),
                                                   ds.shared_prefix))
                                          if ds.shared_prefix else None),
                   "parallelism": f"replicas x{world}",
                   "launch": "cuda graph replay" if args.graph else "direct, programmatic dependent launch",
                   "write": {"fused": "slot mapping fused into the write (one launch)",
                             "attention": "slot mapping and write inside the attention call's "
                                          "first launch",
                             "separate": "slot mapping, then the write"}[args.write]},
        "block_tradeoff": block_tradeoff(step),
        "decode_kv_read_gbs": dec_gbs,
        # the same bytes over decode + combine time (both kernels of split-KV)
        "decode_combine_kv_read_gbs": (work["decode_kv_bytes"] / ((per_kernel[2] + per_kernel[3]) * 1e-3)
                                       / 1e9 if per_kernel[2] > 0 else None),
        # K/V rows as the requests see them (a shared block once per reader):
        # differs from decode_kv_read_gbs only when decode rows share blocks
        "decode_kv_logical_gbs": (work["decode_kv_logical_bytes"] / (dec_ms * 1e-3) / 1e9
                                  if dec_ms > 0 else None),
        # cache write: each new token's K and V rows read and written
        "kv_write": {"kernel": "kv_write_kernel (pkv_paged_kv_write, slots given)",
                     "us": write_ms[0] * 1e3,
                     "gbs": work["write_bytes"] / (write_ms[0] * 1e-3) / 1e9 if write_ms[0] > 0 else None,
                     "us_back_to_back": write_ms[1] * 1e3,
                     "gbs_back_to_back": (work["write_bytes"] / (write_ms[1] * 1e-3) / 1e9
                                          if write_ms[1] > 0 else None),
                     "mapped_us_back_to_back": write_ms[2] * 1e3,
                     "mapped_gbs_back_to_back": (work["write_bytes"] / (write_ms[2] * 1e-3) / 1e9
                                                 if write_ms[2] > 0 else None)},
        "kernel_ms": {"plan": per_kernel[0], "prefill": per_kernel[1],
                      "decode": per_kernel[2], "combine": per_kernel[3]},
        # a step of decodes only: the K/V bytes over every attention kernel
        # (with a shared-prefix hint the tensor-core kernel attends the shared
        # keys, the decode kernel the rest)
        "attention_kv_read_gbs": (work["decode_kv_bytes"] / (sum(per_kernel[1:4]) * 1e-3) / 1e9
                                  if step.max_query_len == 1 else None),
        "roofline": roofline,
        "prefill_roofline": prefill,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * kernels_per_step(step, ds.fused_write, ds.shared_prefix,
                                             ds.write_in_attention),
        "clocks": clocks,
    }
    if rank == 0:
        print(json.dumps(line))
    if pg is not None:
        pg.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_native(args)


if __name__ == "__main__":
    sys.exit(main())
