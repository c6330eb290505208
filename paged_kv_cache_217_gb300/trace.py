"""Per-CTA phase timeline of one decode call (diagnostic).

    python -m paged_kv_cache_217_gb300.build --define PKV_TRACE=1 --out-dir DIR
    python -m paged_kv_cache_217_gb300.trace --lib DIR/libpaged_kv.so --workload llama3_8b

Runs the named layer's decode on the grid kernels (one CTA per sequence, KV
head and partition; --partition -1 by default, or a split-K partition size;
with --planned the step's launch plan is made once, before the traced calls),
with seeded synthetic inputs, blocks scattered through a shuffled pool and L2
evicted between calls, with a trace buffer set
(pkv_set_trace_buffer) and GPU clock stamps (pkv_trace_stamp) before and
after each call, and summarises: where a call's time goes (stamp to first
CTA start, first CTA start to last CTA end, last CTA end to the next stamp;
means over the calls after two warm-up calls), then for the last call the
mean, median, p90 and max of each phase of a CTA's life, CTAs resident per
microsecond, and the phases by tile count. Needs a library built with
PKV_TRACE=1; timings of traced calls are not benchmark numbers.

--calibrate (any build; --lib optional) instead times, between CUDA events
with L2 evicted before each launch, the layer's decode call, an empty
one-CTA kernel, and an empty kernel with the decode grid's CTA count and the
given threads and shared memory (pkv_trace_empty_grid; the defaults are the
tensor-core kernel's 3 warps and bf16 d=128 rings), plus two clock stamps
with nothing between: what any launch of that shape costs before and after
its work, next to the call.

    python -m paged_kv_cache_217_gb300.trace --calibrate --workload llama3_8b --planned

--replay also fits the traced CTA lifetimes as a + b * tiles and replays
the layer's CTAs through as many slots as were resident, rows dispatched in
order, for several row orders (natural; long first; long first and short
last; descending), printing each order's modelled span: a model of the
dispatch only, in which a CTA's life does not depend on its neighbours.
"""

import argparse
import os

import numpy as np

PHASES = ["order (sequence known)", "length and block ids", "first tile landed", "tile loop", "merge and exit"]

# The library's bucket thresholds (kLongFirstX2, kShortLastX8 in csrc/decode.cuh):
# long when 2 * tiles * S >= LONG_FIRST_X2 * total, short when
# 8 * tiles * S <= SHORT_LAST_X8 * total.
LONG_FIRST_X2 = 4
SHORT_LAST_X8 = 5


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--lib", help="a libpaged_kv.so built with PKV_TRACE=1 (optional with --calibrate)")
    ap.add_argument("--workload", default="llama3_8b", choices=["tiny", "llama13b", "llama3_8b", "opt175b_long"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--calls", type=int, default=20)
    ap.add_argument("--partition", type=int, default=-1,
                    help="-1 (one CTA per sequence and KV head) or a split-K partition size in tokens; the "
                         "persistent schedules record no trace")
    ap.add_argument("--planned", action="store_true",
                    help="make the step's launch plan once (pkv_paged_attention_plan) and trace the planned decode "
                         "call, as bench.py times it")
    ap.add_argument("--replay", action="store_true", help="replay the CTA lifetimes under other row orders")
    ap.add_argument("--calibrate", action="store_true",
                    help="time the decode call next to empty launches of its grid's shape (no trace needed)")
    ap.add_argument("--threads", type=int, default=96, help="--calibrate: threads per CTA of the empty grid")
    ap.add_argument("--smem", type=int, default=50224,
                    help="--calibrate: dynamic shared memory (bytes) per CTA of the empty grid")
    args = ap.parse_args(argv)

    import torch
    from . import binding as B
    from . import workloads as W
    if args.lib:
        B.LIB_PATH = os.path.abspath(args.lib)
    elif not args.calibrate:
        raise SystemExit("--lib is required unless --calibrate is given")
    if not args.calibrate and not B.trace_enabled():
        raise SystemExit(f"{args.lib} was not built with PKV_TRACE=1")

    dev = torch.device("cuda", 0)
    shape = W.CONFIGS[args.workload](args.seed)
    lens = shape.context_lens
    nb = W.pool_size(lens, shape.pool_factor)
    tables, _ = W.scattered_tables(lens, nb, args.seed)
    hq, hkv, d = shape.num_q_heads, shape.num_kv_heads, shape.head_dim
    k_pool = W.normal_values((nb, hkv, 16, d), shape.dtype, args.seed * 11 + 1, dev)
    v_pool = W.normal_values((nb, hkv, 16, d), shape.dtype, args.seed * 11 + 2, dev)
    q = W.normal_values((lens.size, hq, d), shape.dtype, args.seed * 11 + 4, dev)
    out = torch.empty_like(q)
    t_d = torch.from_numpy(tables).to(dev)
    l_d = torch.from_numpy(lens).to(dev)
    records = 1 << 17
    buf = torch.zeros(8 * records, dtype=torch.int64, device=dev)
    flush = torch.ones((512 << 20) // 4, dtype=torch.int32, device=dev)
    stamps = torch.zeros(2, dtype=torch.int64, device=dev)
    anatomy = []
    if args.planned:
        B.paged_attention_plan(l_d, t_d, hq, hkv, d, partition_size=args.partition)
    if args.calibrate:
        def decode():
            B.paged_attention_decode(out, q, k_pool, v_pool, t_d, l_d, shape.scale, partition_size=args.partition,
                                     planned=args.planned)
        calibrate(args, shape, decode, flush, stamps, lens.size * hkv)
        return
    B.set_trace_buffer(buf)
    try:
        for i in range(args.calls):
            buf.zero_()
            flush.sum()
            B.trace_stamp(stamps, 0)
            B.paged_attention_decode(out, q, k_pool, v_pool, t_d, l_d, shape.scale, partition_size=args.partition,
                                     planned=args.planned)
            B.trace_stamp(stamps, 1)
            torch.cuda.synchronize()
            r = buf.view(-1, 8).cpu().numpy()
            r = r[r[:, 0] > 0]
            s0, s1 = stamps.cpu().numpy()
            if i >= 2:
                anatomy.append(((r[:, 0].min() - s0) / 1e3, (r[:, 5].max() - r[:, 0].min()) / 1e3,
                                (s1 - r[:, 5].max()) / 1e3))
    finally:
        B.set_trace_buffer(None)
    if anatomy:
        pre, span, post = np.mean(anatomy, axis=0)
        print(f"{shape.name}: stamp -> first CTA {pre:.2f} us, CTA span {span:.2f} us, "
              f"last CTA -> stamp {post:.2f} us (means of {len(anatomy)} calls)")
    t0 = r[:, 0].min()
    st = (r[:, :6] - t0) / 1000.0
    tiles = r[:, 7] >> 32
    d_ph = np.diff(st, axis=1)
    life = st[:, 5] - st[:, 0]
    print(f"{shape.name}: {len(r)} CTAs traced, span {st[:, 5].max():.1f} us")
    for i, name in enumerate(PHASES):
        x = d_ph[:, i]
        print(f"  {name:24s} mean {x.mean():6.2f} us  median {np.median(x):6.2f}  p90 {np.percentile(x, 90):6.2f}"
              f"  max {x.max():6.2f}")
    print(f"  {'lifetime':24s} mean {life.mean():6.2f} us  median {np.median(life):6.2f}"
          f"  p90 {np.percentile(life, 90):6.2f}  max {life.max():6.2f}")
    print(f"  tiles per CTA: mean {tiles.mean():.1f}, max {tiles.max()}")
    grid = np.arange(0.0, st[:, 5].max(), 1.0)
    resident = [int(np.sum((st[:, 0] <= t) & (st[:, 5] > t))) for t in grid]
    print("  CTAs resident per us:", " ".join(map(str, resident)))
    for lo, hi in [(1, 4), (4, 8), (8, 16), (16, 32), (32, 64), (64, 1 << 30)]:
        m = (tiles >= lo) & (tiles < hi)
        if m.any():
            print(f"  tiles [{lo}, {hi if hi < 1 << 30 else 'inf'}): {m.sum():5d} CTAs, life {life[m].mean():6.2f} us,"
                  f" first tile {d_ph[m, 2].mean():5.2f}, loop {d_ph[m, 3].mean():6.2f}, merge {d_ph[m, 4].mean():5.2f}")

    if args.replay:
        replay(tiles, life, lens, shape.num_kv_heads, max(resident) if resident else 1)


def calibrate(args, shape, decode, flush, stamps, ctas):
    """Event-timed medians (and means) over args.calls launches, L2 evicted
    before each launch and outside the events."""
    import torch
    from . import binding as B
    dev = flush.device
    calls = max(args.calls, 20)

    def timed(fn):
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(calls)]
        for i in range(calls + 3):
            flush.sum()
            if i >= 3:
                ev[i - 3][0].record()
            fn()
            if i >= 3:
                ev[i - 3][1].record()
        torch.cuda.synchronize()
        t = np.array([a.elapsed_time(b) * 1e3 for a, b in ev])
        return np.median(t), t.mean()

    rows = [("decode call" + (" (planned)" if args.planned else ""), decode),
            ("empty kernel, 1 CTA x 32 threads", lambda: B.trace_empty_grid(dev, 1, 32, 0)),
            (f"empty kernel, {ctas} CTAs x {args.threads} threads, {args.smem} B shared",
             lambda: B.trace_empty_grid(dev, ctas, args.threads, args.smem))]
    for name, fn in rows:
        med, mean = timed(fn)
        print(f"{shape.name}: {name}: median {med:.2f} us, mean {mean:.2f} us ({calls} launches)")
    gaps = []
    for _ in range(calls):
        flush.sum()
        B.trace_stamp(stamps, 0)
        B.trace_stamp(stamps, 1)
        torch.cuda.synchronize()
        s0, s1 = stamps.cpu().numpy()
        gaps.append((s1 - s0) / 1e3)
    print(f"{shape.name}: stamp -> stamp with nothing between: median {np.median(gaps):.2f} us")
    if B.device_status(clear=True):
        raise SystemExit("device checks tripped during the calibration")


def modelled_span(order, seq_tiles, heads, slots, a, b):
    """End time of CTAs dispatched row by row (all heads of a row's sequence)
    into `slots` slots, each living a + b * tiles."""
    import heapq
    free = [0.0] * slots
    end = 0.0
    for s in order:
        for _ in range(heads):
            t = heapq.heappop(free)
            e = t + a + b * float(seq_tiles[s])
            end = max(end, e)
            heapq.heappush(free, e)
    return end


def replay(tiles, life, lens, heads, slots):
    """Modelled span of the layer under several row orders (the thresholds of
    the library's buckets: long >= 2x the mean tile count, short <= 5/8)."""
    b, a = np.polyfit(tiles.astype(float), life, 1)
    t = (lens.astype(np.int64) + 15) // 16
    S, total = t.size, int(t.sum())
    bucket = [0 if 2 * t[s] * S >= LONG_FIRST_X2 * total else (2 if 8 * t[s] * S <= SHORT_LAST_X8 * total else 1)
              for s in range(S)]
    nat = list(range(S))
    orders = [("natural", nat),
              ("long first", [s for s in nat if bucket[s] == 0] + [s for s in nat if bucket[s] != 0]),
              ("long first, short last", [s for k in (0, 1, 2) for s in nat if bucket[s] == k]),
              ("descending", sorted(nat, key=lambda s: -t[s]))]
    print(f"  replay: life = {a:.2f} + {b:.3f} x tiles us, {slots} slots, {heads} CTAs a sequence")
    for name, order in orders:
        print(f"    {name:28s} modelled span {modelled_span(order, t, heads, slots, a, b):6.2f} us")
    print(f"    {'all slots busy to the end':28s} {(a * S + b * total) * heads / slots:6.2f} us")

if __name__ == "__main__":
    main()
