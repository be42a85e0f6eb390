"""fp64 CPU oracle for prefix-shared KV attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the library imports this package; only the tests, the
smoke check and the benchmark's CPU-baseline leg may call it.  It shares no code with the CUDA
path: it is written from the definitions on the source pages, plainly and slowly, in float64.

Modules
-------
attention   page-1 pool scatter, extend (prefill with a cached prefix) and decode attention as the
            plain softmax(q K^T * scale) V definition, and the log-sum-exp merge of partitions.
radix       longest cached prefix of a token sequence and the token saving at a match unit.
accounting  the pages' closed forms: compute reduction, BatchLLM token-saving ratio, cache hit
            rate and the DFS-optimal hit rate.

Every function is pinned by tests against values the pages print, closed forms, invariants and
brute force on tiny inputs; none is "parity unpinned".
"""
from . import attention, radix, accounting  # noqa: F401
