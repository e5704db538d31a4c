"""Oracle for single-token decode attention over a block-paged KV cache.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may use it.  It shares no code with the CUDA library (no kernels,
headers, helpers, tables or constants) and never receives a value that the
CUDA path computed.

Everything here is plain, slow and written to be checked by eye against the
pages it follows:

* ``attention``  decode attention ``softmax(q.K^T * scale).V`` in float64 over a
  contiguous per-sequence cache, the full causal recompute it must agree with,
  and the paged form that first gathers blocks through a block table.
* ``cache``      the paged pool as plain arrays: slot-mapped append, block copy,
  and a block manager (free list, reference counts, fork, copy-on-write).
* ``fp8``        OCP FP8-E4M3 encoding/decoding from its bit-level definition.

Sources (web pages, cited by title and section):
  [KV Cache篇]           "大模型推理加速——KV Cache篇"
  [KV缓存机制解析]       "KV缓存机制解析：优化大型语言模型推理性能"
  [gptmini 键值缓存]     gptmini "从神经元到GPT" — 键值缓存 chapter
  [PagedAttention]       "KV Cache与PagedAttention：大模型推理显存优化方案"

Pins (tests/test_oracle_*.py, all ``-m "not gpu"``): the worked 4-dim example of
[KV Cache篇] §2.1 in exact arithmetic, closed-form special cases, the
cached = last-row-of-recompute invariant, paged = contiguous under block
permutations, a float64 cross-check against torch's SDPA, brute-force FP8
rounding, and the allocator's closed forms from [PagedAttention] §2.2/§5.1.
No oracle function is "parity unpinned".
"""

from . import attention, cache, fp8  # noqa: F401
