"""CPU oracle for the PagedAttention decode path.

This package is TEST INFRASTRUCTURE. It is a plain, slow, obviously correct
restatement of what the path computes, written in NumPy float64 (and plain
Python for the block manager). Only the test suite, the smoke check of the
graft entry point and the CPU-baseline leg of the benchmark may import it.
The product path (the CUDA library and its Python binding) never imports it,
and this package imports nothing from the product.

Sources (web pages on PagedAttention, cited by title and section):

* "PagedAttention（ページドアテンション）" glossary entry (jisaku.com),
  sections "PagedAttentionの解決策" (16-token blocks, block table
  logical->physical, the 100-token example with table [3, 7, 1, ...]) and
  "コピーオンライト（Copy-on-Write）共有" (parallel sampling, n=3).
* "数万トークンでもVRAMが溢れない！LLM推論を爆速化する「PagedAttention」の全貌"
  (hubblespacetelescope blog), section "OSの知恵をGPUへ" (on-demand blocks,
  waste only in the last block, at most 15 slots; sharing by refcount).
* abeam.tech summary of "Efficient Memory Management for Large Language Model
  Serving with PagedAttention", sections "用語解説" (block table,
  Copy-on-Write), "技術の仕組み / KV キャッシュマネージャ" (fill the last
  block, allocate a new one when full, return blocks on finish),
  "並列サンプリングやビームサーチでの共有" (copy only when a write hits a
  shared block) and "よくある質問" (not a new attention formula).
* "【PagedAttention】とは？" (pro-knowledge-base.com), FAQ on accuracy: paging
  does not change the computed result.

Modules:
  attention      -- decode attention as the plain definition (gather, fp64 softmax)
  cache_ops      -- reshape_and_cache and copy_blocks as element-wise copies
  block_manager  -- independent model of the block manager (free list,
                    refcounts, fork, append with copy-on-write, free)
  numerics       -- exact fp16/bf16 -> fp64 conversion
  quant          -- INT8 KV cache: per-row quantisation, quantised cache
                    write, decode over the dequantised cache
  memsim         -- memory-utilisation replay: paged blocks against
                    contiguous pre-allocation (slot-by-slot arena)

Every function here is pinned by tests in ``tests/test_oracle*.py`` against
values and invariants that the pages and mathematics fix (hand-worked
examples under ``tests/golden/``, brute force on tiny inputs, closed forms,
permutation invariance, copy-on-write sibling equality).
"""

from . import numerics, attention, cache_ops, block_manager, quant, memsim  # noqa: F401
