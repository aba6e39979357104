"""CPU oracle for the PagedWeight fused mixed-precision MoE layer.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The product library never calls
it and shares no code with it; the two meet only in the seeded inputs of
``synthetic/``.

Everything is plain numpy in float64 and follows the definitions on the PagedWeight
pages (arXiv 2607.16184 "PagedWeight: Efficient MoE LLM Serving with Dynamic
Quality-Aware Weight Quantization"):

* ``ap``      -- bit-plane codes, centroid lookup and resident bytes (Sec. 2.2, Sec. 3.1, Eq. 3)
* ``moe``     -- router, top-K, expert FFN and routing-weighted combine (Sec. 2.1, Sec. 3.3)
* ``planner`` -- Eqs. 1, 2, 4-8 and the greedy planner step (Sec. 3.2, Algorithm 1)
* ``pages``   -- the offload / reload ordering of weight pages (Sec. 3.1, Sec. 3.3, Fig. 4)
* ``kv``      -- KV-block accounting coupled to the weight pages: the free-block count F_blk
  of Eq. 7 from the budget the weights leave, the blocks held and the pending growth
  (Sec. 3.2, Sec. 3.3)

Parity status: ``ap`` and ``moe`` are pinned by closed forms, hand-worked examples and
brute force; ``planner`` is pinned for Eqs. 1, 2, 4, 6, 7, 8 and a hand-sorted greedy
example, and its stage/cap policy and reload policy -- readings of Algorithm 1 with no
printed numbers -- by invariants that hold on any input.  ``kv`` is pinned by a
hand-worked sequence from its readings (the pages give the signals, not a formula).
"""
