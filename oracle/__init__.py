"""Plain, slow CPU oracle for paged decode attention.

TEST INFRASTRUCTURE ONLY. Nothing in the product package
(``paged_kv_cache_163_gb300``) imports, links or runs this package; only
``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline arm of
``bench.py`` use it.  It shares no code, table or constant generator with
the CUDA path.

What it computes, and where the pages state it:

* ``allocator``  -- the block manager: 16-token physical blocks allocated on
  demand, a per-sequence block table, prefix blocks shared between
  sequences with copy-on-write, blocks freed when a request finishes
  ("KV Cache 与 vLLM" (zwxr.cn) §3.1-§3.4; "KV Cache优化实战" §4.2).
* ``fp8``        -- the OCP FP8 E4M3 codec used by the FP8 KV cache
  ("KV Cache优化实战" §3.3, ``--kv-cache-dtype fp8_e4m3``).
* ``cache``      -- the paged cache itself: reshape-and-cache writes with an
  optional per-(token, KV-head) absmax FP8 scale ("KV Cache优化实战" §3.2),
  whole-block copies for copy-on-write, and the gather of one sequence's
  blocks through its table into contiguous K/V ("KV Cache 与 vLLM" §3.2).
* ``attention``  -- decode attention softmax(q K^T * scale) V in fp64
  ("企业官网建设流程全解析" (KV Cache 原理篇) §1.2), the split /
  log-sum-exp merge model, a brute-force loop form and the full causal
  recompute that caching must reproduce ("KV Cache 与 vLLM" §1.2-§1.3).
* ``sizing``     -- the pages' KV-size closed forms, utilisation and
  capacity arithmetic.
* ``model``      -- ties the above together to play a workload's operation
  script (create / fork / append / free / decode).

Everything is fp64 (NumPy) except where the method fixes fp32: the FP8 scale
and the division before encoding, which the pages leave open and which are
read as IEEE fp32 round-to-nearest so that codes can be compared bit for bit.
"""
