"""Benchmark of the PagedAttention decode hot path on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload llama13b|llama3_8b|opt66b_sampling|opt175b_long|llama13b_beam|tiny]
                    [--kv native|int8] [--window W]

One step is one pass of the whole hot path over one batch: write each
sequence's new K/V into its slot (reshape_and_cache), the step's launch plan
(pkv_paged_attention_plan: the order in which the decode grid takes the
sequences, made once per step for every layer of the step), and paged
attention decode over every sequence with that plan (split-K decode plus its
log-sum-exp merge when the partition choice splits). The decode figures
(``roofline``, ``per_config``) time the decode call alone; the step figures
(``value``) include the cache write and the plan.
Inputs are synthetic (seeded N(0, 1) values, log-normal/uniform lengths,
blocks scattered through a shuffled pool) with the shapes of the named model
layers. The headline workload is the largest one-GPU configuration, the
OPT-175B-shaped long-context layer (batch 8, 96 heads MHA, head_dim 128, fp16,
lengths uniform in [16384, 32768], blocks scattered through a shuffled pool).
The same run also times the decode call of the LLaMA-13B, Llama-3-8B and
OPT-66B parallel-sampling layers and reports each against the HBM roofline
(``per_config``). The sampling batch (and the beam-search batch), whose
sibling sequences share their prompt blocks, runs the shared-prefix schedule
(partition_size -5: each group of siblings reads its shared blocks once, its
prefix plan made once per step); its roofline figure counts each shared
block once (unique bytes), with the per-sequence (logical) figure beside it.

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
sample of the same workload and reports the same metric. The oracle is split
over the host's cores by KV heads (and, when there are more cores than KV
heads, by sequences): each core runs it unchanged on its share. The
``cpu_baseline`` of this library's arm times the oracle on one sample twice,
on one thread and on all cores.
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
                  "paged_kv_cache_217_gb300/csrc/decode_prefix.cuh",
                  "paged_kv_cache_217_gb300/csrc/cache_ops.cu",
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


def build_workload(name, seed, device, kv="native", window=0, max_seqs=0):
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
        if max_seqs > 0:   # profiling a smaller case of the same layer
            lens = lens[:max_seqs]
        nb = W.pool_size(lens, shape.pool_factor)
        tables, mb = W.scattered_tables(lens, nb, seed)
        k_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 1, device)
        v_pool = W.normal_values((nb, hkv, 16, d), dtype, seed * 11 + 2, device)
        wl.description = shape.name + (f" (first {lens.size} sequences)" if max_seqs > 0 else "")
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


def plan(wl, B):
    """The decode step's launch plan (pkv_paged_attention_plan): made once per
    step, it serves the decode of every layer of that step."""
    if wl.planned:
        B.paged_attention_plan(wl.lens, wl.tables, wl.hq, wl.hkv, wl.d, partition_size=wl.partition)


def decode(wl, B):
    if wl.kv == "int8":
        B.paged_attention_decode_int8(wl.out, wl.q, wl.k_cache, wl.v_cache, wl.k_scale, wl.v_scale, wl.tables,
                                      wl.lens, wl.scale, partition_size=wl.partition, planned=wl.planned)
    elif wl.window > 0:
        B.paged_attention_decode_sliding(wl.out, wl.q, wl.k_pool, wl.v_pool, wl.tables, wl.lens, wl.scale,
                                         wl.window, partition_size=wl.partition)
    else:
        B.paged_attention_decode(wl.out, wl.q, wl.k_pool, wl.v_pool, wl.tables, wl.lens, wl.scale,
                                 partition_size=wl.partition, planned=wl.planned)


def step(wl, B):
    """One pass of the hot path on device-resident inputs."""
    cache_write(wl, B)
    plan(wl, B)
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


def oracle_sample(wl, budget_s, max_pool_bytes=1 << 30):
    """A bounded sample of the workload for the CPU oracle: whole sequences (all
    heads) in workload order until about budget_s seconds of single-thread
    oracle work (at least one sequence, and no more once the gathered pool
    reaches max_pool_bytes), with the used blocks gathered into a small pool
    (table relabelled to match)."""
    import torch
    from paged_kv_cache_217_gb300 import workloads as W
    row_bytes = wl.d + 4 if wl.kv == "int8" else wl.d * 2
    seqs, est_s, pool_bytes = [], 0.0, 0
    for s in range(wl.num_seqs):
        L = int(wl.lens_h[s])
        if wl.window > 0:
            L = min(L, wl.window)
        est_s += L * wl.hkv * ORACLE_S_PER_TOKEN_HEAD + 2e-4 * wl.hq
        pool_bytes += -(-int(wl.lens_h[s]) // 16) * 16 * wl.hkv * row_bytes * 2
        seqs.append(s)
        if est_s >= budget_s or pool_bytes >= max_pool_bytes:
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
        ks = vs = None
    tab = np.full((len(seqs), wl.tables_h.shape[1]), -1, np.int32)
    for i, s in enumerate(seqs):
        nb = -(-int(wl.lens_h[s]) // 16)
        tab[i, :nb] = [remap[int(b)] for b in wl.tables_h[s, :nb]]
    q = W.to_numpy_storage(wl.q_h[seqs], wl.dtype)
    lens = wl.lens_h[seqs]
    attended = np.minimum(lens, wl.window) if wl.window > 0 else lens
    return dict(q=q, kp=kp, vp=vp, ks=ks, vs=vs, tab=tab, lens=lens, seqs=len(seqs),
                bytes=int(attended.astype(np.int64).sum()) * wl.hkv * row_bytes * 2)


# rough single-thread cost of the oracle per (token, KV head): two row gathers
# plus the fp64 math (measured about 1.4e-6 s on the GPU machine's host; kept
# pessimistic so a sample never overruns its budget)
ORACLE_S_PER_TOKEN_HEAD = 4e-6


def host_cores():
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def _shares(sample, hkv, cores):
    """Splits the sample over at most `cores` workers: KV heads into
    min(cores, hkv) contiguous ranges, then, with cores to spare, sequences
    into cores // that many ranges of about equal tokens. Attention of one (sequence, KV head) does not
    depend on any other, so each share is a complete oracle problem."""
    n_h = max(1, min(cores, hkv))
    n_s = max(1, min(cores // n_h, sample["seqs"]))
    h_cuts = [round(i * hkv / n_h) for i in range(n_h + 1)]
    tok = np.cumsum(sample["lens"].astype(np.int64))
    total = int(tok[-1]) if tok.size else 0
    s_cuts = [0] + [int(np.searchsorted(tok, total * i / n_s, side="left")) + 1 for i in range(1, n_s)] + \
        [sample["seqs"]]
    s_cuts = sorted(set(min(max(c, 0), sample["seqs"]) for c in s_cuts))
    out = []
    for h0, h1 in zip(h_cuts[:-1], h_cuts[1:]):
        for s0, s1 in zip(s_cuts[:-1], s_cuts[1:]):
            if h1 > h0 and s1 > s0:
                out.append((h0, h1, s0, s1))
    return out


_WORKER = r"""
import sys, time
import numpy as np
sys.path.insert(0, %(root)r)
import oracle.attention as OA, oracle.quant as OQ
z = np.load(%(path)r)
a = [z[k] for k in %(names)s]
print("ready", flush=True)
for _ in range(%(repeats)d):
    sys.stdin.readline()
    t0, p0 = time.time(), time.perf_counter()
    %(call)s(*a, %(scale)r, %(hkv)d, %(dtype)r%(extra)s)
    print(t0, time.time(), time.perf_counter() - p0, flush=True)
"""


def time_oracle(wl, sample, repeats, cores=1):
    """Runs the oracle `repeats` times on the sample, split over `cores`
    single-threaded worker processes (fresh interpreters: no CUDA state is
    inherited), each running the oracle unchanged on its share. All workers
    load their share first; each repeat then starts them together, and its
    time is the wall time from the first start to the last finish. Returns
    (seconds of each repeat, number of workers)."""
    G = wl.hq // wl.hkv
    shares = _shares(sample, wl.hkv, cores)
    if wl.kv == "int8":
        names, call = "('q', 'kp', 'vp', 'ks', 'vs', 'tab', 'lens')", "OQ.paged_attention_decode_int8"
    else:
        names = "('q', 'kp', 'vp', 'tab', 'lens')"
        call = "OA.paged_attention_decode_window" if wl.window > 0 else "OA.paged_attention_decode"
    extra = f", {int(wl.window)}" if (wl.window > 0 and wl.kv != "int8") else ""
    env = dict(os.environ, OMP_NUM_THREADS="1", OPENBLAS_NUM_THREADS="1", MKL_NUM_THREADS="1")
    procs = []
    with tempfile.TemporaryDirectory() as td:
        try:
            for i, (h0, h1, s0, s1) in enumerate(shares):
                path = os.path.join(td, f"share{i}.npz")
                arrs = dict(q=sample["q"][s0:s1, h0 * G:h1 * G], kp=sample["kp"][:, h0:h1],
                            vp=sample["vp"][:, h0:h1], tab=sample["tab"][s0:s1], lens=sample["lens"][s0:s1])
                if wl.kv == "int8":
                    arrs.update(ks=sample["ks"][:, h0:h1], vs=sample["vs"][:, h0:h1])
                np.savez(path, **{k: np.ascontiguousarray(v) for k, v in arrs.items()})
                code = _WORKER % dict(root=ROOT, path=path, names=names, repeats=repeats, call=call,
                                      scale=wl.scale, hkv=h1 - h0, dtype=wl.dtype, extra=extra)
                procs.append(subprocess.Popen([sys.executable, "-c", code], stdin=subprocess.PIPE,
                                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True,
                                              env=env))
            for p in procs:
                if p.stdout.readline().strip() != "ready":
                    raise RuntimeError(f"oracle worker failed: {p.stderr.read()[-300:]}")
            walls = []
            for _ in range(repeats):
                for p in procs:
                    p.stdin.write("go\n")
                    p.stdin.flush()
                marks = []
                for p in procs:
                    ln = p.stdout.readline().split()
                    if len(ln) != 3:
                        raise RuntimeError(f"oracle worker failed: {p.stderr.read()[-300:]}")
                    marks.append((float(ln[0]), float(ln[1]), float(ln[2])))
                if len(procs) == 1:
                    walls.append(marks[0][2])
                else:
                    walls.append(max(m[1] for m in marks) - min(m[0] for m in marks))
            for p in procs:
                p.stdin.close()
                p.wait(timeout=60)
        finally:
            for p in procs:
                if p.poll() is None:
                    p.kill()
    return walls, len(shares)


def describe_sample(wl, sample, secs, workers):
    how = "1 thread" if workers == 1 else f"{workers} single-threaded processes (one per core, split by KV heads" + \
        (" and sequences)" if workers > wl.hkv else ")")
    return (f"{sample['seqs']} of {wl.num_seqs} sequences (all {wl.hq} heads, {int(sample['lens'].sum())} "
            f"tokens, {sample['bytes'] / 1e6:.1f} MB KV) through the fp64 NumPy oracle, {how}, "
            f"{secs:.4g} s per pass")


def cpu_baseline(wl, budget_s=12.0):
    """The oracle on one bounded sample of the workload, on one thread and on
    every host core (the same sample split by KV heads)."""
    sample = oracle_sample(wl, budget_s)
    secs = time_oracle(wl, sample, 1)[0][0]
    cores = host_cores()
    line = {"value": round(sample["bytes"] / secs / 1e9, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": describe_sample(wl, sample, secs, 1),
            "seqs_layers_per_s": round(sample["seqs"] / secs, 3)}
    if cores > 1:
        walls, workers = time_oracle(wl, sample, 2, cores)
        par = min(walls)
        line["all_cores"] = {"value": round(sample["bytes"] / par / 1e9, 5), "unit": "GB/s", "cores": workers,
                             "host_cores": cores, "os_cpu_count": os.cpu_count(),
                             "sample": describe_sample(wl, sample, par, workers),
                             "seqs_layers_per_s": round(sample["seqs"] / par, 3)}
    return line


# ---------------------------------------------------------------------------
# arms
# ---------------------------------------------------------------------------
PER_CONFIG = ["llama13b", "llama3_8b", "opt66b_sampling", "opt175b_long"]
# Batches whose sibling sequences share prompt blocks run the shared-prefix
# schedule (partition_size -5): each group of siblings reads its shared blocks
# once. Every other workload takes the library's choice (0).
SHARED_PREFIX_WORKLOADS = ("opt66b_sampling", "llama13b_beam")


def default_partition(name, kv, window, B):
    return B.SHARED_PREFIX if name in SHARED_PREFIX_WORKLOADS and window == 0 else 0


def launches_per_step(wl, B):
    """This library's kernels in one step: the cache write, the decode (its
    split-K merge runs inside it), and the one-CTA kernel that orders the
    batch -- the step's launch plan (full attention, either cache; batches of
    2..1024 sequences in grids of at most 4096 CTAs; the prefix plan of the
    shared-prefix schedule), or, for sliding windows, the ordering that the
    decode call itself launches for batches of 128..1024 sequences (see
    pkv_paged_attention_decode). Sets wl.planned."""
    part = B.resolved_partition(wl.num_seqs, wl.hq, wl.hkv, wl.d, wl.tables_h.shape[1], wl.partition)
    if part == B.SHARED_PREFIX:   # the prefix plan, made once per step
        wl.planned = wl.window == 0
        return part, 3
    parts = 1 if part in (-1, B.BALANCED) else -(-wl.tables_h.shape[1] * 16 // part)
    fits = part != B.BALANCED and wl.num_seqs <= 1024 and wl.num_seqs * wl.hkv * parts <= 4096
    wl.planned = wl.window == 0 and fits and wl.num_seqs >= 2
    ordered = wl.planned or (fits and wl.num_seqs >= 128)
    return part, 2 + (1 if ordered else 0)


def time_steps(wl, B, K, flush, stream):
    """K steps on device-resident inputs, L2 evicted (a read of `flush`)
    before each, outside the events. Returns the per-step event times (ms) of
    the whole step and of the decode call."""
    import torch
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True),
           torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    for k in range(K):
        flush.sum()                                   # evict L2 with clean lines between steps
        e_start, e_mid, e_end = ev[k]
        e_start.record(stream)
        cache_write(wl, B)
        plan(wl, B)
        e_mid.record(stream)
        decode(wl, B)
        e_end.record(stream)
    torch.cuda.synchronize()
    return [a.elapsed_time(c) for a, _, c in ev], [b.elapsed_time(c) for _, b, c in ev]


def roofline_figures(wl, dec_ms, peak):
    """Decode-call throughput on the bytes HBM must move: every attended token's
    K and V once, and for batches whose sequences share prompt blocks each
    shared block once (unique bytes); the per-sequence (logical) figure, which
    counts L2 hits of shared blocks as well, goes beside it."""
    hbm_bytes = wl.unique_kv_bytes or wl.kv_bytes
    achieved = hbm_bytes / (dec_ms * 1e-3) / 1e9
    fig = {"achieved": round(achieved, 1), "frac": round(achieved / peak, 4),
           "pct_of_nominal_8000GBs": round(100 * achieved / NOMINAL_HBM_GBS, 2),
           "algorithmic_bytes_per_launch": hbm_bytes,
           "bytes_counted": "unique (each shared block once)" if wl.unique_kv_bytes else "every attended token"}
    if wl.unique_kv_bytes:
        fig["logical_bytes_per_launch"] = wl.kv_bytes
        fig["achieved_logical"] = round(wl.kv_bytes / (dec_ms * 1e-3) / 1e9, 1)
    return fig


def traffic_key(name, kv, window):
    return name + ("" if kv == "native" else f"-{kv}") + (f"-w{window}" if window > 0 else "")


def per_config_entry(name, args, device, B, flush, stream, peak):
    import torch
    wl = build_workload(name, args.seed, device, args.kv, 0)
    wl.partition = default_partition(name, args.kv, 0, B)
    device_inputs(wl, device)
    part, _ = launches_per_step(wl, B)
    for _ in range(max(3, args.warmup)):
        step(wl, B)
    torch.cuda.synchronize()
    _, dec = time_steps(wl, B, args.per_config_steps, flush, stream)
    flags = B.device_status(clear=True)
    if flags:
        raise RuntimeError(f"device checks tripped on {name}: {B.describe_device_flags(flags)}")
    dec_ms = statistics.mean(dec)
    fig = roofline_figures(wl, dec_ms, peak)
    entry = {"workload": wl.description, "num_seqs": wl.num_seqs, "steps": args.per_config_steps,
             "schedule": schedule_name(part, B), "decode_us": round(dec_ms * 1e3, 2),
             "decode_us_median": round(statistics.median(dec) * 1e3, 2), **fig,
             "traffic": recorded_traffic(traffic_key(name, args.kv, 0)),
             "meets_70pct_of_measured": fig["frac"] >= 0.70,
             "meets_70pct_of_nominal": fig["pct_of_nominal_8000GBs"] >= 70.0}
    del wl
    torch.cuda.empty_cache()
    return entry


def schedule_name(part, B):
    return ("balanced persistent (equal tiles per warp)" if part == B.BALANCED else
            "shared prefix (each group of siblings reads its shared blocks once)" if part == B.SHARED_PREFIX else
            "one pass per (sequence, KV head)" if part == -1 else f"split-K, {part}-token partitions")


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
    wl = build_workload(args.workload, args.seed, device, args.kv, args.window, args.max_seqs)
    wl.partition = (args.partition if args.partition is not None
                    else default_partition(args.workload, args.kv, args.window, B))
    device_inputs(wl, device)
    # L2 eviction buffer: read (not written) between timed steps, so the next
    # step starts with L2 full of clean, unrelated lines and pays no write-backs.
    flush = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device=device)
    part, n_launch = launches_per_step(wl, B)

    for _ in range(args.warmup):
        step(wl, B)
    torch.cuda.synchronize()
    B.device_status(clear=True)

    stream = torch.cuda.current_stream(device)
    K = args.steps
    sampler = ClockSampler(local)
    sampler.start()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = sampler.mark()
    step_ms, decode_ms = time_steps(wl, B, K, flush, stream)
    if world > 1:
        dist.barrier()
    t1 = sampler.mark()
    clocks = sampler.stop(t0, t1)
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
        flush.sum()
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
    fig = roofline_figures(wl, dec_ms, peak)
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
            "schedule": schedule_name(part, B),
            "launch_plan": ("made once per step by pkv_paged_attention_plan (inside the step's events, outside "
                            "the decode call's), used by pkv_paged_attention_decode_planned"
                            + (": the sibling groups of the shared-prefix schedule" if part == B.SHARED_PREFIX
                               else "")) if wl.planned else
                           "none (or made inside the decode call)",
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
            "achieved": fig["achieved"],
            "peak": peak,
            "peak_kind": f"{peak_kind} (copy bandwidth, burst)",
            "unit": "GB/s",
            "frac": fig["frac"],
            "traffic": recorded_traffic(traffic_key(args.workload, args.kv, args.window)),
            **{k: v for k, v in fig.items() if k not in ("achieved", "frac")},
            "decode_ms": round(dec_ms, 5),
        },
        "e2e": {
            "value": round(whole_job_gbs(wl.kv_bytes, e2e_ms, world), 1),
            "unit": "GB/s",
            "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms, 5),
        },
        "gpu_launches": K * n_launch,
        "clocks": clocks,
    }
    if wl.unique_kv_bytes:
        line["config"]["unique_kv_bytes_per_step"] = wl.unique_kv_bytes
        line["unique_bytes_gbs"] = round(world * wl.unique_kv_bytes / (per_step_ms * 1e-3) / 1e9, 1)
    if not args.no_cpu_baseline and world == 1:
        line["cpu_baseline"] = cpu_baseline(wl)
    if not args.no_per_config and world == 1 and args.window == 0:
        # the decode call of every target layer, timed the same way (each
        # workload built, timed and freed in turn; the headline's own figures
        # are reused)
        main_entry = {"workload": wl.description, "num_seqs": wl.num_seqs, "steps": K,
                      "schedule": schedule_name(part, B), "decode_us": round(dec_ms * 1e3, 2),
                      "decode_us_median": round(statistics.median(decode_ms) * 1e3, 2), **fig,
                      "traffic": line["roofline"]["traffic"],
                      "meets_70pct_of_measured": fig["frac"] >= 0.70,
                      "meets_70pct_of_nominal": fig["pct_of_nominal_8000GBs"] >= 70.0}
        keep_main = args.partition is None and args.kv == "native" and args.workload in PER_CONFIG
        del wl
        torch.cuda.empty_cache()
        per = {}
        for name in PER_CONFIG:
            if name == args.workload and keep_main:
                per[name] = main_entry
            else:
                per[name] = per_config_entry(name, args, device, B, flush, stream, peak)
        line["per_config"] = {"peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "configs": per}
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
    cores = host_cores()
    # each step is one pass over a sample sized to about `budget` seconds of
    # wall time on all cores (single-thread estimate x cores)
    budget = min(6.0, max(0.02, args.reference_budget / total))
    sample = oracle_sample(wl, budget * cores, max_pool_bytes=512 << 20)
    walls, workers = time_oracle(wl, sample, total, cores)
    secs = walls[args.warmup:]
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
        "cpu_baseline": {"value": round(gbs, 5), "unit": "GB/s", "cores": workers, "kind": "oracle",
                         "host_cores": cores, "sample": describe_sample(wl, sample, per, workers)},
        "e2e": {"value": round(gbs, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="opt175b_long",
                    choices=["llama13b", "llama3_8b", "opt66b_sampling", "opt175b_long", "llama13b_beam", "tiny"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--window", type=int, default=0,
                    help="sliding-window decode over the last W tokens of each sequence (0 = full attention)")
    ap.add_argument("--kv", choices=["native", "int8"], default="native",
                    help="KV cache storage: native (the workload's fp16/bf16) or int8 codes with row scales")
    ap.add_argument("--partition", type=int, default=None,
                    help="decode schedule: 0 = library choice, -1 = one CTA per (sequence, KV head), -2 = "
                         "balanced, -5 = shared prefix, N = split-K partitions of N tokens (default: -5 for the "
                         "sampling and beam batches, else 0)")
    ap.add_argument("--max-seqs", type=int, default=0,
                    help="profiling only: the first N sequences of a fixed-shape layer's batch (a smaller case "
                         "of the same kernel for ncu captures; not a benchmark configuration)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip timing the decode call of the other target layers (per_config)")
    ap.add_argument("--per-config-steps", type=int, default=100,
                    help="timed steps of each per_config layer")
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
