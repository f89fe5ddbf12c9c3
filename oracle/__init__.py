"""CPU oracle for per-step working-set recall -- TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 restatement of what the recall path computes, written
from "KVMem: Virtualizing Million-Token Agent Workspaces on a Consumer GPU"
(§4.3 Mean-K and Eq. (10); §4.4 execution view, delta working set and
re-RoPE; §5 tiled retrieval) and the RoPE identities of "InferScale: GPU-Native
KV Injection for Personalized LLM Serving" (§2 RoPE background, Theorem 6).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its Python binding) never imports, links or calls anything here, and this
package imports nothing from the product path: the two share no code.  Inputs
come from the seeded generator in ``paged_kv_cache_meank_gb300.workload``
(random draws only) or from the test itself.

Modules:
  kvmem  -- NumPy float64 definitions (RoPE, Mean-K, Eq. (10), selector,
            execution view, tiled scoring, residency diff).
  brute  -- pure-Python loops over the same definitions, for tiny inputs.

Every function here is pinned by a CPU test against something other than
itself (closed forms, invariants, library routines, brute force, hand-worked
fixtures under tests/golden/).
"""
