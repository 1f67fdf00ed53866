"""CPU oracle for paged attention — TEST INFRASTRUCTURE ONLY.

Plain, slow, fp64 restatement of what the paged-KV hot path computes, written
from the pages on continuous batching and PagedAttention:

* ``paging``    — the block table and its CPU-side block allocator with
                  refcounts and copy-on-write ("Batching, Scheduling, and
                  Paging", sections *PagedAttention* and *Block sharing*).
* ``cache``     — writing new tokens into their slots, copying a block, and
                  gathering a sequence's pages back into contiguous K/V.
* ``attention`` — ``softmax(Q K^T / sqrt(d_k)) V`` per request over that
                  request's own tokens ("Deep Dive: continuous batching",
                  section *Selective batching*), for one decode query per
                  sequence and for a causal prompt chunk.
* ``fp8``       — e4m3 pages with per-row scales: quantisation of new rows
                  and decode attention over the dequantised pages.

Only the test-suite, the package's smoke check and the benchmark's CPU
baseline may import this package.  The library never calls it, and it shares
no code with the library: it reads the same memory layout through its own
indexing.
"""

from . import attention, cache, fp8, paging

__all__ = ["attention", "cache", "fp8", "paging"]
