"""Sink + ring-buffer cache of a streaming head, as a pure-Python slot model.

Source: vLLM issue "Could you support Attention Sink?" (vllm-project/vllm #1304).
Its block tables show a 16-slot cache (4 blocks of 4) in two designs:

* Mistral's circular buffer (no sinks): once the cache is full, token 16 takes
  slot 0 and token 17 takes slot 1 -- slot = t mod W.
* the attention-sink variant with 2 sink tokens: tokens 0 and 1 never move,
  token 16 takes slot 2 and token 17 takes slot 3.

The design the issue settles on (its "option 3") keeps the sink tokens in a
block of their own and the streamed tokens in a circular buffer, so nothing is
ever copied. With S sink slots followed by R ring slots that reads as:

    slot(t) = t                      if t < S
            = S + ((t - S) mod R)    otherwise

which gives the sink-variant table for S = 2, R = 14 and Mistral's for S = 0,
R = 16 (pinned by tests/golden/). A slot that no token has reached is empty
(position -1).
"""

from __future__ import annotations

EMPTY = -1


def ring_slot(t: int, S: int, R: int) -> int:
    """Slot that token position ``t`` is written to (sinks pinned, ring for the rest)."""
    if t < 0 or R < 1 or S < 0:
        raise ValueError("need t >= 0, S >= 0, R >= 1")
    if t < S:
        return t
    return S + (t - S) % R


class RingCacheSim:
    """Slot -> token-position model of one sequence's sink + ring cache.

    Optionally carries a payload per slot (the key/value rows of that token),
    written by the same rule, so a decode can read "what the cache holds"."""

    def __init__(self, S: int, R: int):
        if S < 0 or R < 1:
            raise ValueError("need S >= 0, R >= 1")
        self.S, self.R = S, R
        self.pos = [EMPTY] * (S + R)
        self.payload = [None] * (S + R)
        self.n = 0

    def append_one(self, payload=None) -> int:
        """Write token ``n`` (one decode step's worth); returns its slot."""
        t = self.n
        s = ring_slot(t, self.S, self.R)
        self.pos[s] = t
        self.payload[s] = payload
        self.n += 1
        return s

    def append(self, T: int, payloads=None) -> None:
        """Append T tokens one by one (the definition a multi-token append must match)."""
        for k in range(T):
            self.append_one(None if payloads is None else payloads[k])

    def positions(self) -> list:
        return list(self.pos)

    def valid_slots(self) -> list:
        return [s for s, p in enumerate(self.pos) if p != EMPTY]


def ring_positions_after(n: int, S: int, R: int) -> list:
    """Slot contents after n single-token appends, by simulation (no closed form used)."""
    sim = RingCacheSim(S, R)
    sim.append(n)
    return sim.positions()


def append_survivors(n: int, T: int, S: int, R: int) -> list:
    """Tokens of a T-token append at positions n ... n+T-1 that are still in the cache
    when the append ends, found by simulating the T single appends one at a time and
    keeping the tokens whose slot was not overwritten by a later token of the same call."""
    last_writer = {}
    for t in range(n, n + T):
        last_writer[ring_slot(t, S, R)] = t
    return sorted(last_writer.values())


def paged_stream_dead_blocks(n: int, S: int, R: int, block_size: int) -> list:
    """Streaming head kept in a pool of token blocks (token t at row t): the logical
    blocks, among those holding rows [0, n), that a caller may free once n tokens are
    held.

    Source: the same vLLM issue, whose later comment proposes keeping the first block
    as the sink, dropping the blocks in the middle and keeping the recent ones. Read
    here as storage only: a query still sees exactly the tokens the sink + ring cache
    would hold, and those are what ``ring_positions_after`` simulates -- for the query
    at position n - 1 and, as the window only moves forward, for every later one. A
    block can go when it holds none of them; found by checking every block against
    every held position (no closed form)."""
    held = [p for p in ring_positions_after(n, S, R) if p != EMPTY]
    blocks = (n + block_size - 1) // block_size
    return [k for k in range(blocks) if not any(k * block_size <= p < (k + 1) * block_size for p in held)]
