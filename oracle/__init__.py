"""CPU oracle for the paged-attention hot path.  TEST INFRASTRUCTURE ONLY.

Only the test suite, `__graft_entry__.smoke()` and the CPU-baseline leg of
`bench.py` may import, call or run anything in this package.  The library
path (the CUDA kernels and the C ABI in `paged_kv_cache_36_gb300`) never
touches it, and this package imports nothing from the library: the two share
no code.  Inputs come from the seeded generators in `workloads`.

It is plain, slow and meant to be read against the pages:

* `paging`    - slot rule, naive cache scatter, per-request block accounting
* `attention` - dense per-request causal GQA softmax attention in float64
* `rope`      - table-driven rotary embedding of Q and K (a dense rotation
                matrix per token) and its fusion with the cache scatter
* `allocator` - a list-based block allocator with reserve / commit / rollback
* `scheduler` - a list-based continuous-batching scheduler with recompute
                preemption, and the step metadata built from its plan

Pages cited (by title and section):
  AI Infra入门干货总结：大模型是如何高效推理的 (joto.ai blog)
  vLLM 抢占机制源码精读 (xiaolong-dev.me)
  GPT-5 时代大模型推理调度系统深度实战 (ybb.press)
  Chunked Prefill 与 Preemption (llm-glossary.tokens-kit.com)
  显存与调度, ch. 32 (aaai.latere.ai)

What pins each part (tests/test_oracle_*.py, run with -m "not gpu"):
  slot rule       - the worked example on "AI Infra入门干货总结" (block_table
                    [5, 8, 12], block_size 16, position 25 -> slot 137) and a
                    brute-force enumeration of the logical-to-physical map
  block counting  - the tail-waste program on "显存与调度" (lengths
                    [37, 81, 130, 211]) against a token-by-token simulation,
                    0 <= w_i < B, and the 7-token / block-size-4 accounting on
                    "Chunked Prefill 与 Preemption"
  attention       - torch's scaled_dot_product_attention on full prefills,
                    the chunked-equals-full trace on "Chunked Prefill 与
                    Preemption", closed forms, pure-Python brute force
  rope            - complex multiplication by e^{ia} (numpy), unit-vector
                    closed forms, orthogonality, the relative-position
                    property, pass-through of dimensions >= rotary_dim
  allocator       - the conservation law and reserve / commit / rollback
                    protocol of "显存与调度" checked after every transition,
                    telescoping of the incremental block demand
  scheduler       - PARITY UNPINNED: no page prints a scheduler trace.  It is
                    pinned only by hand-derived scenarios that follow the
                    preemption loop on "vLLM 抢占机制源码精读", by invariants
                    (token budget, max_num_seqs, no admission after a
                    preemption, conservation, termination) and by agreement
                    with the independent C++ scheduler.
"""
