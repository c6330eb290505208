"""Benchmark of the PagedAttention decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama13b|llama3_8b|opt66b_sampling|opt175b_long|llama13b_beam|tiny]
                    [--kv native|int8] [--window W]

One step is one pass of the whole hot path over one batch: write each
sequence's new K/V into its slot (reshape_and_cache), copy-on-write block
copies when the step has any, and paged attention decode over every sequence
(split-K decode plus its log-sum-exp merge when the partition choice splits).
Inputs are synthetic (seeded N(0, 1) values, log-normal/uniform lengths,
blocks scattered through a shuffled pool) with the shapes of the named model
layers. The headline workload is the LLaMA-13B-shaped layer (batch 64,
40 heads, head_dim 128, bf16, lengths log-normal median 512 sigma 0.8 clipped
to [16, 2048]).

value = algorithmic KV bytes read per step (sum over sequences of
L * num_kv_heads * head_dim * 2 (K and V) * 2 bytes) / device time per step,
in GB/s, with inputs resident in HBM. L2 is flushed between timed steps
(outside the timed events) and the KV working set is larger than L2.

``--kv int8`` runs the same step over the INT8 KV cache (int8 codes plus one
fp32 scale per row): the write quantises, the decode dequantises on the fly;
its bytes per token and KV head are 2 * (head_dim + 4). ``--window W`` runs
sliding-window decode over each sequence's last W tokens; only those tokens'
bytes count.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas: the path has no exchange step); value = all ranks' bytes / the
slowest rank's time.

``--impl reference`` times the fp64 CPU oracle on the host cores on a bounded
sample of the same workload and reports the same metric.
"""

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "paged decode attn HBM GB/s (% of GB300 peak) and sequences·layers/s"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 8000.0
L2_FLUSH_BYTES = 512 << 20
KERNEL_SOURCES = ["paged_kv_cache_217_gb300/csrc/decode.cuh",
                  "paged_kv_cache_217_gb300/csrc/decode_mma.cuh",
                  "paged_kv_cache_217_gb300/csrc/decode_sk.cuh",
                  "paged_kv_cache_217_gb300/csrc/device_common.cuh",
                  "paged_kv_cache_217_gb300/csrc/decode_launch.cuh",
                  "paged_kv_cache_217_gb300/csrc/decode_mma_int8.cuh",
                  "paged_kv_cache_217_gb300/csrc/decode_int8.cu",
                  "paged_kv_cache_217_gb300/csrc/api.cu"]


# ---------------------------------------------------------------------------
# workloads
# ---------------------------------------------------------------------------
class Workload:
    pass


def kernel_sha():
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def build_workload(name, seed, device, kv="native", window=0):
    import torch
    from paged_kv_cache_217_gb300 import binding as B
    from paged_kv_cache_217_gb300 import workloads as W

    wl = Workload()
    wl.name = name
    if name == "opt66b_sampling":
        trace = W.opt66b_parallel_sampling(seed)
        nb = trace.block_budget()
        bm = B.BlockManager(nb, W.shuffled_free_order(nb, seed))
        plan = W.drive_parallel_sampling(trace, bm)
        hq = hkv = trace.num_kv_heads
        d, dtype = trace.head_dim, trace.dtype
        k_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 1, device)
        v_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 2, device)
        if plan.pairs:
            B.copy_blocks(k_pool, v_pool, torch.tensor(plan.pairs, dtype=torch.int64, device=device))
        slots = np.concatenate([s for _, s in plan.step_slots])
        kt = W.normal_values((slots.size, hkv, d), dtype, seed * 11 + 3, device)
        B.reshape_and_cache(kt, kt, k_pool, v_pool, torch.from_numpy(slots).to(device))
        mb = max(-(-L // 16) for L in plan.final_lens.values())
        tables, lens = bm.block_tables(plan.seq_ids, mb)
        wl.description = (f"OPT-66B-shaped layer decode after parallel sampling: {trace.prompt_lens.size} prompts "
                          f"x n={trace.n} = {len(plan.seq_ids)} seqs, H=72 MHA, d=128, fp16, prompts U[512,1024], "
                          f"tails U[0,256], {len(plan.pairs)} copy-on-write pairs")
        scale = trace.scale
        unique_blocks = len({int(b) for b in tables.reshape(-1) if b >= 0})
        wl.unique_kv_bytes = unique_blocks * hkv * 16 * d * 2 * 2
    elif name == "llama13b_beam":
        trace = W.beam_search_trace(seed)
        nb = trace.block_budget()
        bm = B.BlockManager(nb, W.shuffled_free_order(nb, seed))
        W.beam_start(trace, bm)
        hq, hkv, d, dtype = trace.num_q_heads, trace.num_kv_heads, trace.head_dim, trace.dtype
        k_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 1, device)
        v_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 2, device)
        npairs = 0
        for step in range(1, trace.steps + 1):
            st = W.beam_step(trace, bm, step)
            if st.pairs:
                B.copy_blocks(k_pool, v_pool, torch.tensor(st.pairs, dtype=torch.int64, device=device))
                npairs += len(st.pairs)
            kt = W.normal_values((len(st.beam_ids), hkv, d), dtype, seed * 11 + 100 + step, device)
            B.reshape_and_cache(kt, kt, k_pool, v_pool, torch.from_numpy(st.slots).to(device))
        mb = -(-(int(trace.prompt_lens.max()) + trace.steps) // 16)
        tables, lens = bm.block_tables(st.beam_ids, mb)
        wl.description = (f"{trace.name}: decode over {len(st.beam_ids)} beams after {trace.steps} beam steps "
                          f"({npairs} copy-on-write pairs)")
        scale = trace.scale
        unique_blocks = len({int(b) for b in tables.reshape(-1) if b >= 0})
        wl.unique_kv_bytes = unique_blocks * hkv * 16 * d * 2 * 2
    else:
        shape = W.CONFIGS[name](seed)
        hq, hkv, d, dtype = shape.num_q_heads, shape.num_kv_heads, shape.head_dim, shape.dtype
        lens = shape.context_lens
        nb = W.pool_size(lens, shape.pool_factor)
        tables, mb = W.scattered_tables(lens, nb, seed)
        k_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 1, device)
        v_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 2, device)
        wl.description = shape.name
        scale = shape.scale
        wl.unique_kv_bytes = None
    S = lens.shape[0]
    # the step's new token of every sequence sits at its last position (write, then attend)
    slots = np.array([int(tables[s, (L - 1) // 16]) * 16 + (L - 1) % 16 if L > 0 else -1
                      for s, L in enumerate(lens.tolist())], dtype=np.int64)
    wl.dtype, wl.hq, wl.hkv, wl.d, wl.scale = dtype, hq, hkv, d, scale
    wl.num_seqs = S
    wl.k_pool, wl.v_pool = k_pool, v_pool
    wl.tables_h = np.ascontiguousarray(tables, dtype=np.int32)
    wl.lens_h = np.ascontiguousarray(lens, dtype=np.int32)
    wl.slots_h = slots
    wl.q_h = W.normal_values((S, hq, d), dtype, seed * 11 + 4, "cpu")
    wl.knew_h = W.normal_values((S, hkv, d), dtype, seed * 11 + 5, "cpu")
    wl.vnew_h = W.normal_values((S, hkv, d), dtype, seed * 11 + 6, "cpu")
    wl.kv = kv
    wl.num_blocks = k_pool.shape[0]
    if kv == "int8":
        # synthetic INT8 cache of the same pool shape: uniform codes, row scales
        # about max|x| / 127 of N(0, 1) rows
        del k_pool, v_pool
        wl.k_pool = wl.v_pool = None
        nb = wl.num_blocks
        wl.k_cache = W.int8_codes((nb, hkv, 16, d), seed * 11 + 7, device)
        wl.v_cache = W.int8_codes((nb, hkv, 16, d), seed * 11 + 8, device)
        wl.k_scale = W.row_scales((nb, hkv, 16), seed * 11 + 9, device)
        wl.v_scale = W.row_scales((nb, hkv, 16), seed * 11 + 10, device)
        row_bytes = d + 4
        if wl.unique_kv_bytes:
            wl.unique_kv_bytes = wl.unique_kv_bytes // (d * 2) * row_bytes
    else:
        row_bytes = d * 2
    wl.window = window
    attended = np.minimum(wl.lens_h, window) if window > 0 else wl.lens_h
    wl.kv_bytes = int(attended.astype(np.int64).sum()) * hkv * row_bytes * 2
    return wl


def device_inputs(wl, device):
    """The step's inputs (q, new K/V, tables, lengths, slots) packed in one pinned
    host buffer and one device buffer, so a step's host-to-device transfer is a
    single copy; the device tensors are views into the device buffer."""
    import torch
    items = [("q", wl.q_h), ("knew", wl.knew_h), ("vnew", wl.vnew_h),
             ("tables", torch.from_numpy(wl.tables_h)), ("lens", torch.from_numpy(wl.lens_h)),
             ("slots", torch.from_numpy(wl.slots_h))]
    offs, total = {}, 0
    for name, t in items:
        offs[name] = total
        total += (t.numel() * t.element_size() + 255) // 256 * 256
    wl.pack_host = torch.empty(total, dtype=torch.uint8).pin_memory()
    wl.pack_dev = torch.empty(total, dtype=torch.uint8, device=device)
    for name, t in items:
        n = t.numel() * t.element_size()
        wl.pack_host[offs[name]:offs[name] + n].copy_(t.contiguous().reshape(-1).view(torch.uint8))
        setattr(wl, name, wl.pack_dev[offs[name]:offs[name] + n].view(t.dtype).view(t.shape))
    wl.pack_dev.copy_(wl.pack_host)
    wl.out = torch.empty_like(wl.q)


def cache_write(wl, B):
    if wl.kv == "int8":
        B.reshape_and_cache_int8(wl.knew, wl.vnew, wl.k_cache, wl.v_cache, wl.k_scale, wl.v_scale, wl.slots)
    else:
        B.reshape_and_cache(wl.knew, wl.vnew, wl.k_pool, wl.v_pool, wl.slots)


def decode(wl, B):
    if wl.kv == "int8":
        B.paged_attention_decode_int8(wl.out, wl.q, wl.k_cache, wl.v_cache, wl.k_scale, wl.v_scale, wl.tables,
                                      wl.lens, wl.scale, partition_size=wl.partition)
    elif wl.window > 0:
        B.paged_attention_decode_sliding(wl.out, wl.q, wl.k_pool, wl.v_pool, wl.tables, wl.lens, wl.scale,
                                         wl.window, partition_size=wl.partition)
    else:
        B.paged_attention_decode(wl.out, wl.q, wl.k_pool, wl.v_pool, wl.tables, wl.lens, wl.scale,
                                 partition_size=wl.partition)


def step(wl, B):
    """One pass of the hot path on device-resident inputs."""
    cache_write(wl, B)
    decode(wl, B)


# ---------------------------------------------------------------------------
# measurement helpers
# ---------------------------------------------------------------------------
class ClockSampler:
    """nvidia-smi clock/throttle samples taken while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, local_rank):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [x.strip() for x in vis.split(",") if x.strip()]
        self.gpu_index = ids[local_rank] if local_rank < len(ids) else str(local_rank)
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self):
        return time.time()

    def stop(self, t0, t1):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        inside = [ln for t, ln in self.lines if t0 - 0.05 <= t <= t1 + 0.05] or [ln for _, ln in self.lines[-3:]]
        sm, smax, reasons = [], [], set()
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in inside:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for nm, val in zip(names[1:], parts[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def max_over_ranks(values, device="cpu"):
    """Element-wise maximum of `values` over all ranks of the default process
    group (the slowest rank's times); the values themselves on one rank."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def whole_job_gbs(bytes_per_rank_step, ms_per_step, world):
    """Whole-job throughput: every rank moves bytes_per_rank_step per step and a
    step takes ms_per_step on the slowest rank."""
    return world * bytes_per_rank_step / (ms_per_step * 1e-3) / 1e9


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def recorded_traffic(workload):
    """Per-launch DRAM bytes of the decode kernel from the committed ncu summary,
    valid only while the kernel sources hash to the recorded value."""
    p = os.path.join(ROOT, "profiles", "traffic.md")
    try:
        with open(p) as f:
            text = f.read()
    except OSError:
        return None
    sha = kernel_sha()
    for m in re.finditer(r"^traffic: workload=(\S+) kernel_sha=(\S+) bytes_per_launch=(\d+)", text, re.M):
        if m.group(1) == workload and m.group(2) == sha:
            return int(m.group(3))
    return None


def oracle_sample(wl, budget_s):
    """A bounded sample of the workload for the CPU oracle: whole sequences (all
    heads) in workload order until about budget_s seconds of oracle work, with
    the used blocks gathered into a small pool (table relabelled to match)."""
    import torch
    from paged_kv_cache_217_gb300 import workloads as W
    seqs, est_s = [], 0.0
    for s in range(wl.num_seqs):
        L = int(wl.lens_h[s])
        if wl.window > 0:
            L = min(L, wl.window)
        est_s += L * wl.hkv * ORACLE_S_PER_TOKEN_HEAD + 2e-4 * wl.hq
        seqs.append(s)
        if est_s >= budget_s:
            break
    blocks = sorted({int(b) for s in seqs for b in wl.tables_h[s, :-(-int(wl.lens_h[s]) // 16)]})
    remap = {b: i for i, b in enumerate(blocks)}
    if wl.kv == "int8":
        idx = torch.tensor(blocks if blocks else [0], dtype=torch.int64, device=wl.k_cache.device)
        kp, vp, ks, vs = [x.index_select(0, idx).cpu().numpy() for x in
                          (wl.k_cache, wl.v_cache, wl.k_scale, wl.v_scale)]
    else:
        idx = torch.tensor(blocks if blocks else [0], dtype=torch.int64, device=wl.k_pool.device)
        kp = W.to_numpy_storage(wl.k_pool.index_select(0, idx), wl.dtype)
        vp = W.to_numpy_storage(wl.v_pool.index_select(0, idx), wl.dtype)
        ks = vs = np.zeros(0, np.float32)
    tab = np.full((len(seqs), wl.tables_h.shape[1]), -1, np.int32)
    for i, s in enumerate(seqs):
        nb = -(-int(wl.lens_h[s]) // 16)
        tab[i, :nb] = [remap[int(b)] for b in wl.tables_h[s, :nb]]
    q = W.to_numpy_storage(wl.q_h[seqs], wl.dtype)
    lens = wl.lens_h[seqs]
    row_bytes = wl.d + 4 if wl.kv == "int8" else wl.d * 2
    attended = np.minimum(lens, wl.window) if wl.window > 0 else lens
    return dict(q=q, kp=kp, vp=vp, ks=ks, vs=vs, tab=tab, lens=lens, seqs=len(seqs),
                bytes=int(attended.astype(np.int64).sum()) * wl.hkv * row_bytes * 2)


# rough cost of the oracle per (token, KV head): two row gathers plus the fp64 math
ORACLE_S_PER_TOKEN_HEAD = 4e-6


def time_oracle(wl, sample, repeats):
    """Runs the oracle `repeats` times on the sample in a fresh single-threaded
    process (spawned, so no CUDA state is inherited) and returns the seconds of
    each run."""
    with tempfile.TemporaryDirectory() as td:
        path = os.path.join(td, "sample.npz")
        np.savez(path, q=sample["q"], kp=sample["kp"], vp=sample["vp"], ks=sample["ks"], vs=sample["vs"],
                 tab=sample["tab"], lens=sample["lens"])
        extra = ""
        if wl.kv == "int8":
            names, call = "('q', 'kp', 'vp', 'ks', 'vs', 'tab', 'lens')", "OQ.paged_attention_decode_int8"
        elif wl.window > 0:
            names, call = "('q', 'kp', 'vp', 'tab', 'lens')", "OA.paged_attention_decode_window"
            extra = f", {int(wl.window)}"
        else:
            names, call = "('q', 'kp', 'vp', 'tab', 'lens')", "OA.paged_attention_decode"
        code = ("import sys, time, numpy as np; sys.path.insert(0, %r)\n"
                "import oracle.attention as OA, oracle.quant as OQ\n"
                "z = np.load(%r)\n"
                "a = [z[k] for k in %s]\n"
                "for _ in range(%d):\n"
                "    t = time.perf_counter()\n"
                "    %s(*a, %r, %d, %r%s)\n"
                "    print(time.perf_counter() - t, flush=True)\n") % (
                    ROOT, path, names, repeats, call, wl.scale, wl.hkv, wl.dtype, extra)
        env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
        res = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env,
                             timeout=3600)
        if res.returncode != 0:
            raise RuntimeError(f"oracle run failed: {res.stderr.strip()[-300:]}")
        return [float(x) for x in res.stdout.split()]


def describe_sample(wl, sample, secs):
    return (f"{sample['seqs']} of {wl.num_seqs} sequences (all {wl.hq} heads, {int(sample['lens'].sum())} "
            f"tokens, {sample['bytes'] / 1e6:.1f} MB KV) through the fp64 NumPy oracle, 1 thread, "
            f"{secs:.3f} s per pass")


def cpu_baseline(wl, budget_s=12.0):
    sample = oracle_sample(wl, budget_s)
    secs = time_oracle(wl, sample, 1)[0]
    return {"value": round(sample["bytes"] / secs / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": describe_sample(wl, sample, secs),
            "seqs_layers_per_s": round(sample["seqs"] / secs, 3)}


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch
    import torch.distributed as dist
    from paged_kv_cache_217_gb300 import binding as B
    from paged_kv_cache_217_gb300 import build as build_mod

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build_mod.build()
    if world > 1:
        dist.barrier()
    B.lib()

    if args.window > 0 and args.kv != "native":
        raise SystemExit("--window runs on the native cache only")
    wl = build_workload(args.workload, args.seed, device, args.kv, args.window)
    wl.partition = args.partition
    device_inputs(wl, device)
    # L2 eviction buffer: read (not written) between timed steps, so the next
    # step starts with L2 full of clean, unrelated lines and pays no write-backs.
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    part = B.resolved_partition(wl.num_seqs, wl.hq, wl.hkv, wl.d, wl.tables_h.shape[1], args.partition)
    # reshape_and_cache + decode (the split-K merge runs inside the decode kernel),
    # plus the one-CTA ordering kernel that batches of 128..1024 sequences in
    # grids of at most 4096 CTAs get (see pkv_paged_attention_decode)
    parts = 1 if part in (-1, B.BALANCED) else -(-wl.tables_h.shape[1] * 16 // part)
    ordered = part != B.BALANCED and 128 <= wl.num_seqs <= 1024 and wl.num_seqs * wl.hkv * parts <= 4096
    launches_per_step = 2 + (1 if ordered else 0)

    for _ in range(args.warmup):
        step(wl, B)
    torch.cuda.synchronize()
    B.device_status(clear=True)

    stream = torch.cuda.current_stream(device)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = sampler.mark()
    for k in range(K):
        flush_sum = flush.sum()                                  # evict L2 with clean lines between steps
        e_start, e_mid, e_end = ev[k]
        e_start.record(stream)
        cache_write(wl, B)
        e_mid.record(stream)
        decode(wl, B)
        e_end.record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    t1 = sampler.mark()
    clocks = sampler.stop(t0, t1)
    step_ms = [a.elapsed_time(c) for a, _, c in ev]
    decode_ms = [b.elapsed_time(c) for _, b, c in ev]
    total_ms = float(sum(step_ms))
    flags = B.device_status(clear=True)
    if flags:
        raise RuntimeError(f"device checks tripped: {B.describe_device_flags(flags)}")

    # end to end through the public API with host buffers: H2D of the step's
    # inputs from pinned memory, the calls, D2H of the output
    out_h = torch.empty(wl.q_h.shape, dtype=wl.q_h.dtype).pin_memory()
    h2d = wl.pack_host.numel()
    d2h = out_h.numel() * out_h.element_size()
    Ke = max(1, min(K, 200))
    e2e_ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(Ke)]
    torch.cuda.synchronize()
    for k in range(Ke):
        flush_sum = flush.sum()
        s_, e_ = e2e_ev[k]
        s_.record(stream)
        wl.pack_dev.copy_(wl.pack_host, non_blocking=True)   # q, new K/V, tables, lengths, slots
        step(wl, B)
        out_h.copy_(wl.out, non_blocking=True)
        e_.record(stream)
    torch.cuda.synchronize()
    e2e_ms = sum(s_.elapsed_time(e_) for s_, e_ in e2e_ev) / Ke

    per_step_ms, e2e_ms = max_over_ranks([total_ms / K, e2e_ms], device)
    if rank != 0:
        dist.destroy_process_group()
        return

    peak, peak_kind = measured_peak()
    value = whole_job_gbs(wl.kv_bytes, per_step_ms, world)
    dec_ms = statistics.mean(decode_ms)
    achieved = wl.kv_bytes / (dec_ms * 1e-3) / 1e9
    traffic = recorded_traffic(args.workload + ("" if args.kv == "native" else f"-{args.kv}")
                               + (f"-w{args.window}" if args.window > 0 else ""))
    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(per_step_ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": wl.dtype if wl.kv == "native" else "int8",
        "data": "synthetic (seeded N(0,1) K/V/q; shapes and length distributions of the named layer)"
                + ("; INT8 cache: uniform codes in [-127, 127], fp32 row scales U[0.01, 0.03]"
                   if wl.kv == "int8" else ""),
        "config": {
            "workload": wl.description + (" (INT8 KV cache)" if wl.kv == "int8" else "")
                        + (f" (sliding window {wl.window})" if wl.window > 0 else ""),
            "kv_cache": "int8 codes + fp32 row scales, fp32 math" if wl.kv == "int8" else f"{wl.dtype}",
            "num_seqs": wl.num_seqs,
            "kv_bytes_per_step": wl.kv_bytes,
            "schedule": ("balanced persistent (equal tiles per warp)" if part == B.BALANCED else
                         "one pass per (sequence, KV head)" if part == -1 else f"split-K, {part}-token partitions"),
            "l2": f"KV working set {wl.kv_bytes / 1e6:.0f} MB > 129 MB L2, and L2 flushed "
                  f"(a {L2_FLUSH_BYTES >> 20} MB read) between timed steps outside the timed events",
            "parallelism": "replicas" if world > 1 else "single GPU",
        },
        "seqs_layers_per_s": round(world * wl.num_seqs / (per_step_ms * 1e-3), 1),
        "pct_of_peak": {
            f"{peak_kind}_{peak:.0f}GBs": round(100 * value / world / peak, 2),
            "nominal_8000GBs": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        },
        "roofline": {
            "bound": "hbm",
            "kernel": ("paged_decode_kernel<KvInt8>" if wl.kv == "int8" else "paged_decode_kernel") +
                      " (+ its LSE merge when split)",
            "achieved": round(achieved, 1),
            "peak": peak,
            "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "algorithmic_bytes_per_launch": wl.kv_bytes,
            "decode_ms": round(dec_ms, 5),
        },
        "e2e": {
            "value": round(whole_job_gbs(wl.kv_bytes, e2e_ms, world), 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 5),
        },
        "gpu_launches": K * launches_per_step,
        "clocks": clocks,
    }
    if wl.unique_kv_bytes:
        line["config"]["unique_kv_bytes_per_step"] = wl.unique_kv_bytes
        line["unique_bytes_gbs"] = round(world * wl.unique_kv_bytes / (per_step_ms * 1e-3) / 1e9, 1)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()


def run_reference(args):
    """The fp64 oracle on the host cores, one bounded sample of the workload per step."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if world > 1 and rank != 0:
        return
    import torch
    device = "cuda" if torch.cuda.is_available() else "cpu"
    wl = build_workload(args.workload, args.seed, device, args.kv, args.window)
    total = args.steps + args.warmup
    budget = min(6.0, max(0.02, args.reference_budget / total))
    sample = oracle_sample(wl, budget)
    secs = time_oracle(wl, sample, total)[args.warmup:]
    per = statistics.mean(secs)
    gbs = sample["bytes"] / per / 1e9
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": round(gbs, 5),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(per * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "kv_cache": "int8 codes + fp32 row scales" if wl.kv == "int8" else wl.dtype,
        "data": "synthetic (seeded N(0,1) K/V/q; shapes and length distributions of the named layer)",
        "config": {"workload": wl.description, "num_seqs": wl.num_seqs, "kv_bytes_per_step": wl.kv_bytes,
                   "sample_kv_bytes_per_step": sample["bytes"]},
        "seqs_layers_per_s": round(sample["seqs"] / per, 3),
        "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": describe_sample(wl, sample, per)},
        "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="llama13b",
                    choices=["llama13b", "llama3_8b", "opt66b_sampling", "opt175b_long", "llama13b_beam", "tiny"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window decode over the last W tokens of each sequence (0 = full attention)")
    ap.add_argument("--kv", choices=["native", "int8"], default="native",
                    help="KV cache storage: native (the workload's fp16/bf16) or int8 codes with row scales")
    ap.add_argument("--partition", type=int, default=0,
                    help="decode schedule: 0 = library choice, -1 = one CTA per (sequence, KV head), "
                         "N = split-K partitions of N tokens")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--lib", default=None,
                    help="load this libpaged_kv.so instead of the package's own (a variant built with "
                         "python -m paged_kv_cache_217_gb300.build --out-dir DIR --define NAME=VALUE)")
    ap.add_argument("--reference-budget", type=float, default=150.0,
                    help="seconds of oracle work for the whole reference run (split over its steps)")
    args = ap.parse_args(argv)
    if args.lib:
        from paged_kv_cache_217_gb300 import binding as B
        B.LIB_PATH = os.path.abspath(args.lib)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
