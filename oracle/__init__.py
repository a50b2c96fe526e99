"""CPU oracle for GraniKV decode-step attention.  TEST INFRASTRUCTURE ONLY.

Plain, slow, float64 restatements of what the method computes (``attention``), of its two KV
pools (``allocators``) and of its per-step backend rule (``dispatch``).  Only the tests, the
package's smoke check and the benchmark's CPU-baseline leg may import it; the product path
(the CUDA library and its Python binding) never does, and shares no code with it.
"""
