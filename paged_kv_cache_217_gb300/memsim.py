"""Memory-utilisation simulator: paged KV blocks against contiguous
pre-allocation, replayed over a request-length trace.

The pages contrast two ways of holding the KV cache of running requests:

* contiguous pre-allocation (glossary entry "PagedAttention（ページドアテンション）",
  section "従来の事前割り当て問題"; blog "数万トークンでもVRAMが溢れない！…",
  section "これまでの問題"): at admission a request reserves one contiguous
  span for its maximum length, however short its output turns out; spans of
  different sizes leave holes between them (external fragmentation). The
  abeam.tech summary (section "既存方式はメモリをかなり無駄にしていた")
  reports that only 20.4 %-38.2 % of the KV memory of such systems holds
  token states;
* paged blocks (glossary entry, "PagedAttentionの解決策"; blog,
  "OSの知恵をGPUへ"): 16-token blocks taken on demand as the sequence grows
  and returned when it finishes, so only the last block of a sequence is
  partly empty (at most 15 slots, under 4 % waste).

The simulator runs both over the same trace in decode steps:

1. admission, first come first served, while the head of the queue fits:
   contiguous -- a first-fit span of R = min(max_len, P + max_new_tokens)
   token slots; paged -- ceil(P / 16) free blocks (the block manager's
   add_seq). An admitted request holds its P prompt tokens.
2. decode: every running request, in admission order, appends one token.
   Paged appends go through the block manager's append_slot; when it is out
   of blocks the most recently admitted running request is preempted (its
   blocks freed, back to the queue in arrival order, its progress lost) and
   the append is retried -- unless the preempted request was the appending
   one, which then skips this step.
3. completion: a request with P + O tokens leaves and frees its memory.
4. the step's record: running requests, stored tokens (sum of lengths),
   allocated token slots (contiguous: sum of R; paged: 16 x blocks in use).

Requests that can never fit (contiguous: P + O above R, or R above the
capacity; paged: ceil((P + O) / 16) blocks above the capacity) are rejected
up front. The paged scheme drives the library's C++
block manager; the contiguous arena is a sorted free-span list.
"""

import bisect
from dataclasses import dataclass, field

from . import binding as _B

BLOCK_SIZE = _B.BLOCK_SIZE


@dataclass
class StepRecord:
    running: int
    stored_tokens: int
    allocated_slots: int


@dataclass
class SimResult:
    scheme: str
    capacity_slots: int
    steps: int = 0
    generated_tokens: int = 0     # decode tokens computed, including those lost to preemption
    useful_tokens: int = 0        # output tokens of completed requests
    completed: int = 0
    rejected: int = 0
    preemptions: int = 0
    fragmentation_stalls: int = 0   # admissions refused although enough slots were free in total
    records: list = field(default_factory=list)

    @property
    def utilisation_of_allocated(self):
        """Token states held / token slots allocated, summed over all steps."""
        a = sum(r.allocated_slots for r in self.records)
        return sum(r.stored_tokens for r in self.records) / a if a else 0.0

    @property
    def utilisation_of_capacity(self):
        """Token states held / whole KV capacity, summed over all steps."""
        return sum(r.stored_tokens for r in self.records) / (self.steps * self.capacity_slots) \
            if self.steps else 0.0

    @property
    def mean_batch(self):
        return sum(r.running for r in self.records) / self.steps if self.steps else 0.0

    @property
    def tokens_per_step(self):
        """Output tokens of completed requests per decode step (throughput)."""
        return self.useful_tokens / self.steps if self.steps else 0.0

    def summary(self):
        return {
            "scheme": self.scheme, "steps": self.steps, "completed": self.completed,
            "rejected": self.rejected, "preemptions": self.preemptions,
            "fragmentation_stalls": self.fragmentation_stalls,
            "utilisation_of_allocated": round(self.utilisation_of_allocated, 6),
            "utilisation_of_capacity": round(self.utilisation_of_capacity, 6),
            "mean_batch": round(self.mean_batch, 4), "tokens_per_step": round(self.tokens_per_step, 4),
        }


class _SpanArena:
    """First-fit allocator of contiguous token spans; free spans kept sorted by start."""

    def __init__(self, size):
        self.starts = [0]
        self.lengths = [size]

    def total_free(self):
        return sum(self.lengths)

    def alloc(self, n):
        for i, ln in enumerate(self.lengths):
            if ln >= n:
                start = self.starts[i]
                if ln == n:
                    del self.starts[i], self.lengths[i]
                else:
                    self.starts[i] += n
                    self.lengths[i] -= n
                return start
        return None

    def free(self, start, n):
        i = bisect.bisect_left(self.starts, start)
        self.starts.insert(i, start)
        self.lengths.insert(i, n)
        if i + 1 < len(self.starts) and self.starts[i] + self.lengths[i] == self.starts[i + 1]:
            self.lengths[i] += self.lengths[i + 1]
            del self.starts[i + 1], self.lengths[i + 1]
        if i > 0 and self.starts[i - 1] + self.lengths[i - 1] == self.starts[i]:
            self.lengths[i - 1] += self.lengths[i]
            del self.starts[i], self.lengths[i]


def _blocks(n):
    return -(-n // BLOCK_SIZE)


def simulate(prompt_lens, output_lens, num_blocks, scheme, max_len, max_new_tokens=None,
             free_order=None, max_steps=10_000_000):
    """Replays the trace (request i: prompt_lens[i] prompt tokens, output_lens[i]
    >= 1 generated tokens) on a KV cache of num_blocks 16-token blocks.

    scheme: "paged" or "contiguous". Contiguous reservations are
    min(max_len, P + max_new_tokens) slots (max_new_tokens defaults to
    max_len, i.e. every request reserves max_len). free_order: the paged
    block manager's initial free stack. Returns a SimResult.
    """
    P = [int(x) for x in prompt_lens]
    O = [int(x) for x in output_lens]
    if len(P) != len(O) or any(p < 1 for p in P) or any(o < 1 for o in O):
        raise ValueError("every request needs a prompt and at least one output token")
    if scheme not in ("paged", "contiguous"):
        raise ValueError(f"unknown scheme {scheme!r}")
    cap = num_blocks * BLOCK_SIZE
    max_new = max_len if max_new_tokens is None else int(max_new_tokens)
    reserve = [min(max_len, p + max_new) for p in P]
    res = SimResult(scheme, cap)

    queue = []
    for i in range(len(P)):
        too_big = (P[i] + O[i] > reserve[i] or reserve[i] > cap) if scheme == "contiguous" \
            else _blocks(P[i] + O[i]) > num_blocks
        if too_big:
            res.rejected += 1
        else:
            queue.append(i)

    running = []            # request ids in admission order
    length = {}
    span = {}
    arena = _SpanArena(cap) if scheme == "contiguous" else None
    bm = _B.BlockManager(num_blocks, free_order) if scheme == "paged" else None
    try:
        while queue or running:
            if res.steps >= max_steps:
                raise RuntimeError("simulation did not drain within max_steps")
            # 1. admission
            while queue:
                i = queue[0]
                if scheme == "contiguous":
                    start = arena.alloc(reserve[i])
                    if start is None:
                        if arena.total_free() >= reserve[i]:
                            res.fragmentation_stalls += 1
                        break
                    span[i] = start
                else:
                    if bm.num_free() < _blocks(P[i]):
                        break
                    bm.add_seq(i, P[i])
                queue.pop(0)
                running.append(i)
                length[i] = P[i]
            # 2. decode: one token per running request
            k = 0
            while k < len(running):
                i = running[k]
                if scheme == "paged":
                    appended = False
                    while not appended:
                        try:
                            bm.append_slot(i)
                            appended = True
                        except _B.OutOfBlocks:
                            # preempt the latest admission (possibly i itself)
                            victim = running[-1]
                            if victim == i and len(running) == 1:
                                raise RuntimeError("out of blocks with nothing to preempt")
                            running.pop()
                            bm.free_seq(victim)
                            del length[victim]
                            bisect.insort(queue, victim)
                            res.preemptions += 1
                            if victim == i:
                                break
                    if not appended:
                        continue        # i was the last running request: the loop ends
                length[i] += 1
                res.generated_tokens += 1
                k += 1
            # 3. record, then completion
            stored = sum(length[i] for i in running)
            alloc = sum(reserve[i] for i in running) if scheme == "contiguous" \
                else BLOCK_SIZE * (num_blocks - bm.num_free())
            res.records.append(StepRecord(len(running), stored, alloc))
            res.steps += 1
            still = []
            for i in running:
                if length[i] == P[i] + O[i]:
                    if scheme == "contiguous":
                        arena.free(span.pop(i), reserve[i])
                    else:
                        bm.free_seq(i)
                    del length[i]
                    res.completed += 1
                    res.useful_tokens += O[i]
                else:
                    still.append(i)
            running = still
    finally:
        if bm is not None:
            bm.close()
    return res


def main(argv=None):
    import argparse
    import json

    from . import workloads as W

    ap = argparse.ArgumentParser(description="paged vs contiguous KV memory utilisation on a synthetic trace")
    ap.add_argument("--trace", choices=["llama13b", "llama3_8b"], default="llama13b")
    ap.add_argument("--requests", type=int, default=512)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--capacity-requests", type=int, default=32,
                    help="KV capacity in units of one max-length reservation")
    ap.add_argument("--max-new-tokens", type=int, default=None)
    args = ap.parse_args(argv)
    P, O, max_len = W.memsim_trace(args.trace, args.requests, args.seed)
    num_blocks = args.capacity_requests * max_len // BLOCK_SIZE
    for scheme in ("contiguous", "paged"):
        r = simulate(P, O, num_blocks, scheme, max_len, args.max_new_tokens)
        print(json.dumps(dict(trace=args.trace, requests=args.requests, num_blocks=num_blocks,
                              max_len=max_len, **r.summary())))


if __name__ == "__main__":
    main()
