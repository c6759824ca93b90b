"""CPU oracle for paged decode attention and gather_cached_kv.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or links
anything in this package: only the tests, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` use it.  It shares
no code, tables or helpers with the CUDA library; the seeded input generator
(``paged_kv_decode_22_gb300.workloads``) feeds both sides and holds none of the
arithmetic.

Everything is float64 NumPy (or pure Python for the brute-force reference) and
follows the plain definitions:

* ``paged_attention`` -- decode-phase attention over a paged KV cache, the
  operation the vLLM pages call ``single_query_cached_kv_attention``
  ("Optimizes the single_query_cached_kv_attention kernel", vLLM pull request
  420; MQA/GQA head sharing from "Optimize MQA Kernel", pull request 452).
* ``split_context`` -- the split-context form of the same softmax (partial
  results per context range and their log-sum-exp merge), the idea behind the
  "Paged attention V2" column of the kernel-latency tables in
  "[Performance] Support MQA/GQA in decode phase by using FlashAttention".
* ``gather`` -- ``gather_cached_kv`` from "Memcpy kernel for flash attention"
  (vLLM pull request 29).
* ``cache`` -- writing new tokens' K/V into the pool at a slot mapping (the
  ``cache_ops.cache`` step named in the FlashAttention pull request's notes).
* ``prefill`` -- a chunk of several new query tokens per sequence attending
  causally over the same paged cache (the review comments of the
  FlashAttention pull request: the KV-cache attention kernel serves prefill
  too, with or without a cached prefix); one query per sequence is decode.
* ``brute`` -- triple-loop dense attention on contiguous K/V, for tiny inputs.
"""
