"""Independent model of the memory-utilisation simulation: paged blocks
against contiguous pre-allocation over a request-length trace.

Test infrastructure (see the package docstring). The product's simulator
(which drives the C++ block manager and a free-span arena) is compared with
this model step record by step record.

What the pages fix:
* Contiguous pre-allocation reserves, at admission, one contiguous region for
  a request's maximum length however short its output is, and regions of
  different sizes leave holes (glossary entry "PagedAttention（ページドアテン
  ション）", section "従来の事前割り当て問題", the 4096-token reservation
  example; blog "数万トークンでもVRAMが溢れない！…", section "これまでの問題").
* Paged blocks are taken on demand and returned at the end; only a
  sequence's last block is partly empty (glossary entry,
  "PagedAttentionの解決策"; blog, "OSの知恵をGPUへ").

Readings where the pages are silent (the step rules):
1. Admission, first come first served while the head of the queue fits:
   contiguous -- the lowest-addressed run of R = min(max_len, P +
   max_new_tokens) free slots; paged -- ceil(P / 16) free blocks. The
   admitted request holds its P prompt tokens.
2. Decode: each running request in admission order appends one token. A
   paged append with no block to take preempts the most recently admitted
   running request (freed, requeued in arrival order, progress lost); if that
   was the appending request it skips the step, else the append is retried.
3. Record (running, stored tokens, allocated slots), then requests holding
   P + O tokens finish and free their memory.
Requests that can never fit are rejected before the first step.

The contiguous arena here is a slot-by-slot occupancy list scanned from
address 0; the paged side is the oracle block manager.
"""

from .block_manager import BLOCK_SIZE, OracleBlockManager, OutOfBlocks


def blocks_for(tokens):
    return (tokens + BLOCK_SIZE - 1) // BLOCK_SIZE


def first_free_run(used, n):
    """Lowest start address of n consecutive free slots, or None."""
    run = 0
    for addr, u in enumerate(used):
        run = 0 if u else run + 1
        if run == n:
            return addr - n + 1
    return None


def simulate(prompt_lens, output_lens, num_blocks, scheme, max_len, max_new_tokens=None,
             free_order=None):
    """Returns a dict: steps, records [(running, stored, allocated)], completed,
    rejected, preemptions, fragmentation_stalls, generated_tokens, useful_tokens."""
    P = [int(x) for x in prompt_lens]
    O = [int(x) for x in output_lens]
    cap = num_blocks * BLOCK_SIZE
    if max_new_tokens is None:
        max_new_tokens = max_len
    R = [min(max_len, p + max_new_tokens) for p in P]
    out = dict(steps=0, records=[], completed=0, rejected=0, preemptions=0, fragmentation_stalls=0,
               generated_tokens=0, useful_tokens=0)

    waiting = []
    for i in range(len(P)):
        if scheme == "contiguous":
            never = P[i] + O[i] > R[i] or R[i] > cap
        else:
            never = blocks_for(P[i] + O[i]) > num_blocks
        if never:
            out["rejected"] += 1
        else:
            waiting.append(i)

    used = [False] * cap
    where = {}
    bm = OracleBlockManager(num_blocks, BLOCK_SIZE, free_order)
    running, tokens = [], {}

    while waiting or running:
        # 1. admission
        while waiting:
            i = waiting[0]
            if scheme == "contiguous":
                start = first_free_run(used, R[i])
                if start is None:
                    if used.count(False) >= R[i]:
                        out["fragmentation_stalls"] += 1
                    break
                for a in range(start, start + R[i]):
                    used[a] = True
                where[i] = start
            else:
                if bm.num_free() < blocks_for(P[i]):
                    break
                bm.add_seq(i, P[i])
            waiting.pop(0)
            running.append(i)
            tokens[i] = P[i]

        # 2. decode
        k = 0
        while k < len(running):
            i = running[k]
            skipped = False
            if scheme == "paged":
                while True:
                    try:
                        bm.append_slot(i)
                        break
                    except OutOfBlocks:
                        last = running.pop()
                        bm.free_seq(last)
                        del tokens[last]
                        waiting = sorted(waiting + [last])
                        out["preemptions"] += 1
                        if last == i:
                            skipped = True
                            break
            if skipped:
                continue
            tokens[i] += 1
            out["generated_tokens"] += 1
            k += 1

        # 3. record, then completion
        stored = sum(tokens[i] for i in running)
        if scheme == "contiguous":
            allocated = sum(R[i] for i in running)
        else:
            allocated = BLOCK_SIZE * (num_blocks - bm.num_free())
        out["records"].append((len(running), stored, allocated))
        out["steps"] += 1
        keep = []
        for i in running:
            if tokens[i] == P[i] + O[i]:
                if scheme == "contiguous":
                    for a in range(where[i], where[i] + R[i]):
                        used[a] = False
                    del where[i]
                else:
                    bm.free_seq(i)
                del tokens[i]
                out["completed"] += 1
                out["useful_tokens"] += O[i]
            else:
                keep.append(i)
        running = keep
    return out
