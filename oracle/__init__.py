"""CPU oracle for mixed-head (retrieval / streaming) causal attention and its cache.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The library under
``streaming_kv_cache_duo_gb300`` never imports it and has no CPU fallback.

Plain, slow, float64 restatements of what the pages define:

* ``ring_cache``: the sink + ring-buffer cache (slot of each token, what a cache
  holds after n appends, a multi-token append), from the block tables of the
  vLLM issue "Could you support Attention Sink?".
* ``attention``: the visible-key rule of retrieval and streaming heads from the
  DuoAttention README (Abstract), masked softmax attention in float64 written
  two independent ways (a dense L x L mask, and a per-row gather of the visible
  keys), decode over a cache, chunked prefill against a growing cache, and the
  log-sum-exp merge of partial softmaxes used by the vLLM Dual Chunk Attention
  pull request.
* ``kv4``: the 4-bit KV cache row encoding (asymmetric codes with an fp16 scale and
  zero per row; the README pairs DuoAttention with a 4-bit KV cache but gives no
  format, so this is the plainest reading, stated in the module).
* ``dca``: Dual Chunk Attention from that pull request (three query vectors chosen
  by the chunk of the key relative to the query's, a per-position fp32 scale),
  written as the definition and as the pull request's brute-force schedule.

Every function is pinned by tests in ``tests/test_oracle_*.py`` against the
pages' worked tables (``tests/golden/``), closed forms, brute force and an
independent library routine (torch's scaled_dot_product_attention in float64).
No function here is "parity unpinned".
"""

from .ring_cache import RingCacheSim, ring_slot, ring_positions_after, append_survivors  # noqa: F401
from .attention import (  # noqa: F401
    RETRIEVAL, STREAMING, is_visible, visible_keys, attention_dense_mask, attend_rows,
    prefill, prefill_chunked, decode_from_cache, lse_merge, partial_softmax,
    visible_pair_count,
)
