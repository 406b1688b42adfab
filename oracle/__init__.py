"""Oracle for the paged KV-cache path (decode, chunked prefill, block manager with
prefix caching, beam steps and swapping): plain, slow, obviously correct CPU code.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` may import, call or
execute anything in this package. The product (``paged_kv_cache_259_gb300``) never
imports it, and this package imports nothing from the product: the two share no
kernels, headers, helpers, tables or constant generators. Only the seeded input
generators in ``pkv_workloads`` feed both sides.

Arithmetic is float64 throughout, except where a method step fixes another
precision (the FP8 quantiser divides in float32 and rounds to E4M3, because the
stored byte is decided in that precision).

Sources, by page title and section:

* "PagedAttention" (Ultralytics glossary), section "Cách phân trang hoạt động"
  (how paging works): fixed-size blocks (16 tokens by default), one shared pool,
  a per-request block table, lazy allocation when the last block is full, the
  attention kernel reading keys back through the table, and the worked
  40-token example.
* Same page, section "Chia sẻ block giữa các chuỗi" (sharing blocks): several
  sequences point at one physical block, with a reference count per block, and a
  shared block is copied before a sequence writes into it (copy-on-write).
* Same page, section "Các kỹ thuật liên quan" (related techniques):
  FlashAttention-style tiling, grouped-query attention, FP8 cache quantisation.
* "KV cache paginado e batching contínuo para LLMs" (upskillscore), section
  "Como funciona": block tables, waste confined to the last block, reference
  counts, block-level copy-on-write (allocate another block, copy, decrement the
  original's count); preemption by swapping blocks to CPU memory.
* "vLLM PagedAttention: uma revolução no throughput..." (news.hada.io), the
  feature list: chunked prefill, prefix caching.

Modules:

* ``attention``    -- decode and chunked-prefill attention as the plain softmax
                      definition, over K/V gathered through the block table.
* ``cache_ops``    -- slot-mapped write of new K/V, block copy for copy-on-write,
                      block copy between the device and host pools (swapping).
* ``fp8_e4m3``     -- E4M3 decode/encode written from the OCP FP8 definition.
* ``block_manager``-- free list, block tables, reference counts, fork, CoW, free,
                      beam-search reshuffles, swapping to a host pool, and the
                      script replayer.
* ``prefix_cache`` -- the block manager with full blocks shared across requests
                      by their exact prefix (evictable when unused).
"""
