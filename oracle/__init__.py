"""CPU oracle for the CSA2 FP4 sparse-decode path and the CED KV projection.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only tests/, the smoke check in __graft_entry__ and the CPU-baseline leg of
bench.py may use it. It shares no code with the CUDA library.

Every function is a plain, slow, direct statement of what the method computes,
in float64 NumPy, following the pages of "DeepSeek-V4.1-Flash: Pushing the
Limits of KV Cache Compression" (the picx.dev summary is the only page with the
equations; the blog repost and the abstract add the SWA / sparse combination
and the layer-reuse facts). Where the pages are silent the plainest reading is
taken; each such reading is named in the function that makes it.

Modules:
  fp4        E2M1 codes with one E4M3 scale per 16 channels (table enumeration)
  indexer    multi-head ReLU indexer scores and top-K selection
  attention  sparse MQA over selected entries, sliding window, LSE merge
  ced        CED projection C_l = H W_l^KV, Z_l = H W_l^Z with the FP4 cache write
  decode     one CSA2 layer group (FULL / REINDEX / REUSE) end to end
  append     decode-time cache append (window ring, one FP4 entry every 4 tokens)

Parity status: every function is pinned by tests under tests/test_oracle_*.py
to values the pages or the mathematics fix; the only unpinned item is
whole-model behaviour (it needs trained weights), which is out of scope.
"""
from . import fp4, indexer, attention, ced, decode, append  # noqa: F401
