"""Independent model of the KV block manager, in plain Python.

Test infrastructure (see the package docstring). The C++ block manager in the
product library is compared against this model bit for bit (tables,
refcounts, slots, copy-on-write pairs, free counts) on scripted traces.

What the pages fix:
* Fixed-size physical blocks of 16 tokens and a per-sequence block table of
  physical ids that need not be contiguous (glossary entry,
  "PagedAttentionの解決策"). A 100-token request occupies ceil(100/16) = 7
  blocks and only the last is partly empty.
* Blocks are taken on demand: tokens fill the last block and a new block is
  allocated when it is full; a finished request returns its blocks
  (abeam.tech summary, "KV キャッシュマネージャ"; blog,
  "オンデマンドなブロック割り当て"). Waste is at most 15 slots per sequence,
  in the last block only (blog, "メモリ浪費をほぼ0%").
* Parallel samples of one prompt share the prompt's blocks by reference
  count, without copying (blog, "複数リクエスト間でのブロック共有"); a shared
  block is copied only when a write reaches it (abeam.tech summary,
  "並列サンプリングやビームサーチでの共有"; glossary entry,
  "コピーオンライト（Copy-on-Write）共有", n=3 samples).

Readings where the pages are silent:
* The free list is a stack. It starts as ``initial_free_order`` (bottom at
  index 0); allocation pops from the top (the end); a block whose refcount
  reaches 0 is pushed on top. Within one call, blocks are taken in logical
  order and returned in table order.
* append_slot with L tokens in the sequence: if L is a multiple of 16 (the
  last block is full, or there is none) a new block is allocated; otherwise,
  if the last block's refcount is above 1, the writer copies it: a new block
  is allocated, the pair (last, new) is emitted, the old block's refcount
  drops by one and the table's last entry becomes the new block. Full shared
  blocks are never copied, because appends only ever write the last block.
  The slot returned is table[L // 16] * 16 + L % 16 and L becomes L + 1.
* Every failing call raises and leaves the state unchanged.
* Beam search and shared prefixes (abeam.tech summary, "並列サンプリングや
  ビームサーチでの共有" and the evaluation's shared-prefix workloads): a beam
  step forks each new beam from its parent beam and drops the old beams; a
  request whose prompt repeats another request's prefix shares the whole
  blocks of that prefix. Both only move references, never data.
* Sliding window (glossary entry, "他のKVキャッシュ最適化との組み合わせ"
  names sliding-window attention alongside paging): blocks wholly before the
  window are released (release_before); their table entries become -1 so
  that later blocks keep their logical indices.
"""

BLOCK_SIZE = 16


class BlockManagerError(Exception):
    """Base class of the block manager's failures."""


class OutOfBlocks(BlockManagerError):
    """The free list holds fewer blocks than the call needs."""


class InvalidArgument(BlockManagerError):
    """Unknown or duplicate sequence id, bad size or bad block id."""


class OracleBlockManager:
    def __init__(self, num_blocks, block_size=BLOCK_SIZE, initial_free_order=None):
        if num_blocks <= 0 or block_size <= 0:
            raise InvalidArgument("num_blocks and block_size must be positive")
        order = list(range(num_blocks)) if initial_free_order is None \
            else [int(b) for b in initial_free_order]
        if sorted(order) != list(range(num_blocks)):
            raise InvalidArgument("initial_free_order must be a permutation of 0..num_blocks-1")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = order
        self.refcount = [0] * num_blocks
        self.tables = {}
        self.lengths = {}

    # -- queries -------------------------------------------------------------
    def num_free(self):
        return len(self.free)

    def block_table(self, seq_id):
        return list(self.tables[seq_id])

    def length(self, seq_id):
        return self.lengths[seq_id]

    # -- operations ----------------------------------------------------------
    def _need(self, n):
        if n > len(self.free):
            raise OutOfBlocks(f"need {n} blocks, {len(self.free)} free")

    def _pop(self):
        b = self.free.pop()
        self.refcount[b] = 1
        return b

    def add_seq(self, seq_id, num_tokens):
        """A new sequence holding num_tokens tokens: ceil(num_tokens/16) fresh blocks."""
        if seq_id in self.tables:
            raise InvalidArgument(f"sequence {seq_id} exists")
        if num_tokens < 0:
            raise InvalidArgument("num_tokens must be >= 0")
        nb = -(-num_tokens // self.block_size)
        self._need(nb)
        self.tables[seq_id] = [self._pop() for _ in range(nb)]
        self.lengths[seq_id] = num_tokens

    def fork(self, parent, child):
        """child shares every block of parent; each shared block's refcount grows by one."""
        if parent not in self.tables:
            raise InvalidArgument(f"unknown sequence {parent}")
        if child in self.tables:
            raise InvalidArgument(f"sequence {child} exists")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            if b >= 0:                      # released entries (-1) are not shared
                self.refcount[b] += 1

    def append_slot(self, seq_id):
        """Reserve the slot of the next token. Returns (slot, cow_src, cow_dst); -1 = no copy."""
        if seq_id not in self.tables:
            raise InvalidArgument(f"unknown sequence {seq_id}")
        table = self.tables[seq_id]
        L = self.lengths[seq_id]
        src = dst = -1
        if L % self.block_size == 0:
            self._need(1)
            table.append(self._pop())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                self._need(1)
                new = self._pop()
                self.refcount[last] -= 1
                table[-1] = new
                src, dst = last, new
        slot = table[L // self.block_size] * self.block_size + L % self.block_size
        self.lengths[seq_id] = L + 1
        return slot, src, dst

    def free_seq(self, seq_id):
        """Drop the sequence; blocks whose refcount reaches 0 go back on the free list."""
        if seq_id not in self.tables:
            raise InvalidArgument(f"unknown sequence {seq_id}")
        for b in self.tables.pop(seq_id):
            if b < 0:
                continue
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
        del self.lengths[seq_id]

    def beam_reorder(self, old_ids, parents, new_ids):
        """Beam search step: new beam i continues old beam old_ids[parents[i]]
        (a fork: it shares that beam's blocks); afterwards every old beam is
        dropped. Blocks no surviving beam holds go back on the free list (old
        beams in the given order, each in table order). new_ids must be
        distinct and may reuse ids of old beams only. Allocates nothing, so it
        cannot run out of blocks."""
        old_ids = [int(x) for x in old_ids]
        parents = [int(x) for x in parents]
        new_ids = [int(x) for x in new_ids]
        if len(set(old_ids)) != len(old_ids) or any(o not in self.tables for o in old_ids):
            raise InvalidArgument("old beams must be distinct live sequences")
        if len(parents) != len(new_ids) or any(p < 0 or p >= len(old_ids) for p in parents):
            raise InvalidArgument("one parent index into old_ids per new beam")
        if len(set(new_ids)) != len(new_ids) or any(n in self.tables and n not in old_ids for n in new_ids):
            raise InvalidArgument("new beam ids must be distinct and unused")
        children = [(list(self.tables[old_ids[p]]), self.lengths[old_ids[p]]) for p in parents]
        for table, _ in children:
            for b in table:
                if b >= 0:
                    self.refcount[b] += 1
        for o in old_ids:
            self.free_seq(o)
        for n, (table, length) in zip(new_ids, children):
            self.tables[n] = table
            self.lengths[n] = length

    def add_seq_with_prefix(self, seq_id, num_tokens, donor, prefix_tokens):
        """New sequence of num_tokens tokens whose first tokens repeat the first
        prefix_tokens tokens of sequence `donor`: the whole blocks of that
        common prefix are shared with the donor (refcount + 1), the rest are
        fresh blocks. Returns the number of positions shared (a multiple of
        16); the caller writes K/V from that position on."""
        if seq_id in self.tables:
            raise InvalidArgument(f"sequence {seq_id} exists")
        if donor not in self.tables:
            raise InvalidArgument(f"unknown sequence {donor}")
        if num_tokens < 0 or prefix_tokens < 0:
            raise InvalidArgument("num_tokens and prefix_tokens must be >= 0")
        shared = min(prefix_tokens, num_tokens, self.lengths[donor]) // self.block_size
        head = self.tables[donor][:shared]
        if any(b < 0 for b in head):
            raise InvalidArgument("the donor has released blocks of that prefix")
        fresh = -(-num_tokens // self.block_size) - shared
        self._need(fresh)
        for b in head:
            self.refcount[b] += 1
        self.tables[seq_id] = list(head) + [self._pop() for _ in range(fresh)]
        self.lengths[seq_id] = num_tokens
        return shared * self.block_size

    def release_before(self, seq_id, first_token):
        """Sliding window: drop the sequence's hold on every block that lies
        wholly before position first_token (blocks j with (j+1)*16 <=
        first_token), in table order. Their table entries become -1 (logical
        positions keep their blocks' indices); a block whose refcount reaches
        0 goes back on the free list. Returns the number of entries dropped."""
        if seq_id not in self.tables:
            raise InvalidArgument(f"unknown sequence {seq_id}")
        if first_token < 0 or first_token > self.lengths[seq_id]:
            raise InvalidArgument("first_token must be in [0, length]")
        table = self.tables[seq_id]
        dropped = 0
        for j in range(first_token // self.block_size):
            b = table[j]
            if b < 0:
                continue
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)
            table[j] = -1
            dropped += 1
        return dropped

    def padded_tables(self, seq_ids, max_blocks_per_seq):
        """([n][max_blocks_per_seq] table padded with -1, [n] lengths)."""
        rows, lens = [], []
        for s in seq_ids:
            t = self.tables[s]
            if len(t) > max_blocks_per_seq:
                raise InvalidArgument(f"sequence {s} has {len(t)} blocks > {max_blocks_per_seq}")
            rows.append(t + [-1] * (max_blocks_per_seq - len(t)))
            lens.append(self.lengths[s])
        return rows, lens
