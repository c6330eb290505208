"""Seeded synthetic inputs for the decode path (shapes, lengths, tables, values).

This module only draws random inputs. It holds none of the attention or
block-management arithmetic, so both the CUDA path and the CPU oracle can be
fed from it without sharing any of the method's code.

The pages' workloads are serving traces (ShareGPT- and Alpaca-length request
mixes on OPT-13B/66B/175B and LLaMA-13B, abeam.tech summary, "使ったデータセ
ットと評価設定"). Those datasets are not used; the five configurations below
stand in for them with their shapes only: head counts and head_dim of the
named models, log-normal or uniform context lengths, 16-token blocks placed
at random in a shuffled pool, and N(0, 1) values.
"""

from dataclasses import dataclass, field
import math

import numpy as np

BLOCK_SIZE = 16


@dataclass
class DecodeShape:
    """One decode workload: sizes plus per-sequence context lengths."""
    name: str
    dtype: str                 # "f16" or "bf16"
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    context_lens: np.ndarray   # int32 [num_seqs]
    pool_factor: float = 1.2
    scale: float = field(default=None)

    def __post_init__(self):
        if self.scale is None:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def num_seqs(self):
        return int(self.context_lens.shape[0])

    @property
    def elem_bytes(self):
        return 2


def _lognormal_lengths(rng, n, median, sigma, lo, hi):
    x = rng.lognormal(mean=math.log(median), sigma=sigma, size=n)
    return np.clip(np.rint(x), lo, hi).astype(np.int32)


def tiny_decode(seed=0):
    """Batch 4, lengths {5, 17, 33, 64}, 4 q heads = 4 KV heads, head_dim 64, fp16.

    The pool has 64 blocks; the caller assigns them with a seeded permutation.
    """
    del seed
    return DecodeShape("tiny: B=4, H=4, d=64, fp16, L={5,17,33,64}", "f16", 4, 4, 64,
                       np.array([5, 17, 33, 64], dtype=np.int32))


def llama13b_mha_decode(seed=0):
    """LLaMA-13B-shaped layer: 40 heads MHA, head_dim 128, bf16, batch 64,
    lengths log-normal (median 512, sigma 0.8) clipped to [16, 2048]."""
    rng = np.random.default_rng(seed)
    return DecodeShape("LLaMA-13B layer: B=64, Hq=Hkv=40, d=128, bf16, L~logN(512,0.8)",
                       "bf16", 40, 40, 128, _lognormal_lengths(rng, 64, 512, 0.8, 16, 2048))


def llama3_8b_gqa_decode(seed=0):
    """Llama-3-8B-shaped GQA layer: 32 q heads / 8 KV heads, head_dim 128, bf16,
    batch 256, lengths log-normal (median 150, sigma 0.6) clipped to [8, 1024]."""
    rng = np.random.default_rng(seed)
    return DecodeShape("Llama-3-8B layer: B=256, Hq=32, Hkv=8, d=128, bf16, L~logN(150,0.6)",
                       "bf16", 32, 8, 128, _lognormal_lengths(rng, 256, 150, 0.6, 8, 1024))


def opt175b_long_decode(seed=0):
    """OPT-175B-shaped layer: 96 heads MHA, head_dim 128, fp16, batch 8,
    lengths uniform in [16384, 32768]."""
    rng = np.random.default_rng(seed)
    return DecodeShape("OPT-175B layer: B=8, Hq=Hkv=96, d=128, fp16, L~U[16384,32768]",
                       "f16", 96, 96, 128,
                       rng.integers(16384, 32768, size=8, endpoint=True).astype(np.int32))


@dataclass
class ParallelSamplingTrace:
    """Parallel sampling: prompts, n samples each, and each sample's tail length."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prompt_lens: np.ndarray    # int32 [num_prompts]
    tail_lens: np.ndarray      # int32 [num_prompts, n]
    scale: float = field(default=None)

    def __post_init__(self):
        if self.scale is None:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def n(self):
        return int(self.tail_lens.shape[1])

    def block_budget(self, block_size=BLOCK_SIZE):
        """An upper bound on the blocks the trace can hold at once."""
        per_prompt = -(-self.prompt_lens // block_size)
        tails = (-(-(self.tail_lens + block_size) // block_size)).sum(axis=1)
        return int((per_prompt + tails).sum())


def opt66b_parallel_sampling(seed=0, num_prompts=32, n=4, prompt_range=(512, 1024),
                             tail_range=(0, 256)):
    """OPT-66B-shaped layer (72 heads MHA, head_dim 128, fp16): 32 prompts x n=4
    samples, prompt lengths uniform [512, 1024], tails uniform [0, 256]."""
    rng = np.random.default_rng(seed)
    prompts = rng.integers(prompt_range[0], prompt_range[1], size=num_prompts,
                           endpoint=True).astype(np.int32)
    tails = rng.integers(tail_range[0], tail_range[1], size=(num_prompts, n),
                         endpoint=True).astype(np.int32)
    return ParallelSamplingTrace(
        f"OPT-66B layer: {num_prompts} prompts x n={n}, H=72, d=128, fp16", "f16", 72, 72, 128,
        prompts, tails)


CONFIGS = {
    "tiny": tiny_decode,
    "llama13b": llama13b_mha_decode,
    "llama3_8b": llama3_8b_gqa_decode,
    "opt66b_sampling": opt66b_parallel_sampling,
    "opt175b_long": opt175b_long_decode,
}


def memsim_trace(name, num_requests, seed=0):
    """A request-length trace for the memory-utilisation simulator: total
    lengths L from the named layer's length distribution, each split into a
    prompt of ceil(L / 2) tokens and an output of the rest; with the
    distribution's upper clip as the maximum length. Returns (prompt_lens,
    output_lens, max_len)."""
    rng = np.random.default_rng(seed)
    if name == "llama13b":
        L, max_len = _lognormal_lengths(rng, num_requests, 512, 0.8, 16, 2048), 2048
    elif name == "llama3_8b":
        L, max_len = _lognormal_lengths(rng, num_requests, 150, 0.6, 8, 1024), 1024
    else:
        raise ValueError(f"unknown trace {name!r}")
    P = (L + 1) // 2
    return P.astype(np.int64), (L - P).astype(np.int64), max_len


def shuffled_free_order(num_blocks, seed):
    """A seeded random permutation of the physical block ids 0..num_blocks-1."""
    return np.random.default_rng(seed + 1_000_003).permutation(num_blocks).astype(np.int32)


def pool_size(context_lens, pool_factor=1.2, block_size=BLOCK_SIZE):
    """Blocks in the pool: pool_factor times the blocks the sequences occupy."""
    used = int((-(-np.asarray(context_lens, dtype=np.int64) // block_size)).sum())
    return max(1, int(math.ceil(pool_factor * used)))


def scattered_tables(context_lens, num_blocks, seed, block_size=BLOCK_SIZE, extra_cols=0):
    """Block tables that place each sequence's blocks at random pool positions.

    Sequence s takes the next ceil(L_s / block_size) ids of a seeded
    permutation of the pool. Returns (int32 [S, max_blocks] padded with -1,
    max_blocks). ``extra_cols`` widens the table (unused columns stay -1).
    """
    lens = np.asarray(context_lens, dtype=np.int64)
    nbs = -(-lens // block_size)
    if int(nbs.sum()) > num_blocks:
        raise ValueError("pool too small for the sequences")
    order = shuffled_free_order(num_blocks, seed)
    max_blocks = max(1, int(nbs.max()) if lens.size else 1) + extra_cols
    tables = np.full((lens.size, max_blocks), -1, dtype=np.int32)
    pos = 0
    for s, nb in enumerate(nbs.tolist()):
        tables[s, :nb] = order[pos:pos + nb]
        pos += nb
    return tables, max_blocks


def normal_values(shape, dtype, seed, device="cpu"):
    """A torch tensor of N(0, 1) values rounded to fp16 or bf16, drawn with a
    seeded generator on ``device`` (values differ between devices)."""
    import torch
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.normal_(generator=gen)
    return x.to(tdt)


def int8_codes(shape, seed, device="cpu"):
    """A torch int8 tensor of codes drawn uniformly from [-127, 127] with a
    seeded generator on ``device`` (the synthetic content of an INT8 cache)."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    return torch.randint(-127, 128, shape, generator=gen, dtype=torch.int8, device=device)


def row_scales(shape, seed, device="cpu", lo=0.01, hi=0.03):
    """A torch float32 tensor of per-row scales drawn uniformly from [lo, hi]
    (about max|x| / 127 for rows of N(0, 1) values), seeded on ``device``."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    x = torch.empty(shape, dtype=torch.float32, device=device)
    x.uniform_(lo, hi, generator=gen)
    return x


def to_numpy_storage(t, dtype):
    """Host NumPy view of a 16-bit tensor: float16 for fp16, uint16 bits for bf16."""
    import torch
    t = t.detach().cpu().contiguous()
    if dtype == "f16":
        return t.numpy()
    return t.view(torch.int16).numpy().view(np.uint16)


@dataclass
class SamplingPlan:
    """What driving a block manager through a ParallelSamplingTrace produced."""
    seq_ids: list               # sample s of prompt i has id i * n + s
    prompt_of: list             # prompt index of each sequence
    step_slots: list            # per decode step: (seq ids appending, int64 slots)
    pairs: list                 # copy-on-write (src, dst) pairs, in emission order
    final_lens: dict            # seq id -> tokens after the tails


def drive_parallel_sampling(trace, bm):
    """Runs the parallel-sampling script against any block manager with
    add_seq / fork / append_slot: add each prompt as sample 0, fork samples
    1..n-1 from it, then decode the tails one step at a time; in each step
    every sequence whose tail is not finished appends one token, in
    ascending sequence id."""
    n = trace.n
    seq_ids, prompt_of = [], []
    for i, plen in enumerate(trace.prompt_lens.tolist()):
        root = i * n
        bm.add_seq(root, plen)
        seq_ids.append(root)
        prompt_of.append(i)
        for c in range(1, n):
            bm.fork(root, root + c)
            seq_ids.append(root + c)
            prompt_of.append(i)
    tails = {i * n + c: int(trace.tail_lens[i, c]) for i in range(trace.prompt_lens.shape[0])
             for c in range(n)}
    steps, pairs = [], []
    for step in range(int(trace.tail_lens.max()) if trace.tail_lens.size else 0):
        active = [sid for sid in seq_ids if tails[sid] > step]
        slots = np.empty(len(active), dtype=np.int64)
        for j, sid in enumerate(active):
            slot, src, dst = bm.append_slot(sid)
            slots[j] = slot
            if src >= 0:
                pairs.append((src, dst))
        steps.append((active, slots))
    final = {sid: int(trace.prompt_lens[sid // n]) + tails[sid] for sid in seq_ids}
    return SamplingPlan(seq_ids, prompt_of, steps, pairs, final)


@dataclass
class BeamSearchTrace:
    """Beam search: prompts, a beam width, and per step the parent beam of
    every new beam (a seeded, skewed choice: a few strong beams tend to
    survive, as in beam search)."""
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    prompt_lens: np.ndarray    # int32 [num_prompts]
    parents: np.ndarray        # int32 [steps, num_prompts, width]
    scale: float = field(default=None)

    def __post_init__(self):
        if self.scale is None:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def width(self):
        return int(self.parents.shape[2])

    @property
    def steps(self):
        return int(self.parents.shape[0])

    def block_budget(self, block_size=BLOCK_SIZE):
        """An upper bound on the blocks the trace can hold at once: every beam
        private from the prompt's last block on, plus the prompt."""
        per_beam = -(-(self.steps + block_size) // block_size) + 1
        return int((-(-self.prompt_lens // block_size)).sum() + self.prompt_lens.size * self.width * per_beam)


def beam_search_trace(seed=0, num_prompts=16, width=4, steps=64, prompt_range=(512, 1024),
                      num_heads=40, head_dim=128, dtype="bf16"):
    """LLaMA-13B-shaped layer (40 heads MHA, head_dim 128, bf16): 16 prompts of
    U[512, 1024] tokens, beam width 4, 64 beam steps."""
    rng = np.random.default_rng(seed)
    prompts = rng.integers(prompt_range[0], prompt_range[1], size=num_prompts, endpoint=True).astype(np.int32)
    weights = np.array([2.0 ** -i for i in range(width)])
    weights /= weights.sum()
    parents = np.sort(rng.choice(width, size=(steps, num_prompts, width), p=weights), axis=2).astype(np.int32)
    return BeamSearchTrace(f"LLaMA-13B layer beam search: {num_prompts} prompts x width {width}, {steps} steps, "
                           f"H=40, d=128, bf16, prompts U[{prompt_range[0]},{prompt_range[1]}]", dtype,
                           num_heads, num_heads, head_dim, prompts, parents)


@dataclass
class BeamStep:
    beam_ids: list             # beams after the step's reorder, prompt-major
    slots: np.ndarray          # int64 slot of each beam's new token
    pairs: list                # copy-on-write (src, dst) pairs of the step's appends


def beam_ids(trace, step):
    """Beam ids alive after `step` reorders (step 0 = the initial fork)."""
    return [(i * (trace.steps + 1) + step) * trace.width + j for i in range(trace.prompt_lens.size)
            for j in range(trace.width)]


def beam_start(trace, bm):
    """Adds every prompt and forks it into `width` beams (any block manager with
    add_seq / fork / free_seq). Returns the initial beam ids."""
    ids = beam_ids(trace, 0)
    for i, plen in enumerate(trace.prompt_lens.tolist()):
        root = ids[i * trace.width]
        bm.add_seq(root, plen)
        for j in range(1, trace.width):
            bm.fork(root, ids[i * trace.width + j])
    return ids


def beam_step(trace, bm, step):
    """Step `step` (1-based) of the script: each prompt's beams are reordered by
    the trace's parents, then every beam appends one token (append_slot, in
    beam order). Returns a BeamStep."""
    old, new = beam_ids(trace, step - 1), beam_ids(trace, step)
    w = trace.width
    for i in range(trace.prompt_lens.size):
        bm.beam_reorder(old[i * w:(i + 1) * w], trace.parents[step - 1, i].tolist(), new[i * w:(i + 1) * w])
    slots = np.empty(len(new), dtype=np.int64)
    pairs = []
    for k, sid in enumerate(new):
        slot, src, dst = bm.append_slot(sid)
        slots[k] = slot
        if src >= 0:
            pairs.append((src, dst))
    return BeamStep(new, slots, pairs)
