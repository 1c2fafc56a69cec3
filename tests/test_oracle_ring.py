"""Pins of the oracle's sink + ring cache model (CPU only)."""

import os

import pytest

import oracle
import oracle.ring_cache as rc
from oracle import RingCacheSim, ring_slot, append_survivors

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load_table(name):
    meta, events = {}, []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line.startswith("# sink_size"):
                parts = line[2:].replace(",", "").split()
                meta = {"S": int(parts[1]), "slots": int(parts[3])}
            if not line or line.startswith("#"):
                continue
            tok = line.split()
            events.append((tok[0], [-1 if x == "x" else int(x) for x in tok[1:]]))
    return meta, events


def _replay(meta, events):
    """Fill the cache to the table's initial state, then one append per later row."""
    S = meta["S"]
    R = meta["slots"] - S
    sim = RingCacheSim(S, R)
    got = []
    for k, (name, _) in enumerate(events):
        if k == 0:
            sim.append(sum(1 for x in events[0][1] if x >= 0))
        else:
            sim.append_one()
        got.append(sim.positions())
    return got


@pytest.mark.parametrize("name", ["mistral_ring_S0_16slots.txt", "sink_ring_S2_16slots.txt"])
def test_block_tables_from_the_page(name):
    meta, events = _load_table(name)
    got = _replay(meta, events)
    for (ev, want), have in zip(events, got):
        assert have == want, (name, ev)


def test_page_events_slots():
    # the sink table: token 16 -> slot 2, token 17 -> slot 3; Mistral's: 16 -> 0, 17 -> 1
    assert ring_slot(16, 2, 14) == 2 and ring_slot(17, 2, 14) == 3
    assert ring_slot(16, 0, 16) == 0 and ring_slot(17, 0, 16) == 1


def test_planted_slot_mistake_fails_the_tables(monkeypatch):
    # A plausible mistake (wrapping over all S + R slots, which moves the sinks)
    # must break the sink table while still passing Mistral's (S = 0).
    monkeypatch.setattr(rc, "ring_slot", lambda t, S, R: t % (S + R))
    meta, events = _load_table("sink_ring_S2_16slots.txt")
    got = _replay(meta, events)
    assert any(h != w for (_, w), h in zip(events, got))


@pytest.mark.parametrize("S,R", [(0, 1), (0, 5), (1, 1), (2, 14), (4, 32), (3, 7), (64, 256)])
def test_contents_after_n_appends(S, R):
    # After n appends the cache holds exactly [0, min(n,S)) U [max(S, n-R), n), each once.
    for n in list(range(0, 2 * (S + R) + 3)) + [1000, 1001]:
        pos = oracle.ring_positions_after(n, S, R)
        held = sorted(p for p in pos if p >= 0)
        want = sorted(set(range(min(n, S))) | set(range(max(S, n - R), n)))
        assert held == want, (n, S, R)
        assert len(pos) == S + R
        # each held token sits at its own slot
        for s, p in enumerate(pos):
            if p >= 0:
                assert ring_slot(p, S, R) == s
        # empty slots are exactly a suffix [n, S + R) while the cache is not full
        assert pos.count(-1) == max(0, S + R - n)


@pytest.mark.parametrize("S,R", [(0, 3), (2, 5), (4, 32), (64, 256)])
def test_multi_token_append_survivors(S, R):
    for n in [0, 1, S, S + 1, S + R - 1, S + R, 3 * (S + R) + 1]:
        for T in [1, 2, R - 1, R, R + 1, S + R + 5, 3 * R + 2]:
            if T < 1:
                continue
            surv = append_survivors(n, T, S, R)
            want = [t for t in range(n, n + T) if t < S or t >= n + T - R]
            assert surv == want
            # writing only the survivors gives the same state as T single appends
            a = RingCacheSim(S, R)
            a.append(n)
            for t in surv:
                a.pos[ring_slot(t, S, R)] = t
            b = RingCacheSim(S, R)
            b.append(n + T)
            assert a.pos == b.pos
            # no two survivors share a slot
            assert len({ring_slot(t, S, R) for t in surv}) == len(surv)


def test_invalid_parameters():
    with pytest.raises(ValueError):
        RingCacheSim(2, 0)
    with pytest.raises(ValueError):
        ring_slot(-1, 2, 3)


# --------------------------------------------------- block-granular eviction (paged pool)
def _held(n, S, R):
    return [p for p in rc.ring_positions_after(n, S, R) if p >= 0]


@pytest.mark.parametrize("S,R,bs", [(0, 16, 4), (2, 14, 4), (4, 32, 8), (64, 256, 128), (5, 3, 4), (130, 1, 128)])
def test_dead_blocks_closed_form(S, R, bs):
    # past the sink blocks, and ending at or before the window of the last token
    for n in range(0, 6 * (S + R + bs)):
        lo = -(-S // bs)
        hi = max(lo, max(0, n - R) // bs)
        assert rc.paged_stream_dead_blocks(n, S, R, bs) == list(range(lo, hi)), n


@pytest.mark.parametrize("S,R,bs", [(0, 16, 4), (2, 14, 4), (3, 5, 4), (64, 256, 128)])
def test_dead_blocks_never_hold_a_visible_token_and_only_grow(S, R, bs):
    prev = set()
    for n in range(1, 4 * (S + R + bs)):
        dead = set(rc.paged_stream_dead_blocks(n, S, R, bs))
        # every key the query at n - 1 or a later query can see is in a kept block
        q = n - 1
        for j in range(n):
            if j < S or q - j < R:
                assert j // bs not in dead
        # a block dropped once stays dropped; the kept blocks are exactly those of held tokens
        assert prev <= dead
        prev = dead
        kept = set(range(-(-n // bs))) - dead
        assert kept == {p // bs for p in _held(n, S, R)}


def test_dead_blocks_special_cases():
    # window covering everything: nothing to drop; R = 1, no sinks: all but the last token's block
    assert rc.paged_stream_dead_blocks(100, 0, 1000, 16) == []
    assert rc.paged_stream_dead_blocks(100, 0, 1, 16) == list(range(6))
    # sinks only reach into block 0: the blocks between it and the window go
    assert rc.paged_stream_dead_blocks(100, 4, 20, 16) == [1, 2, 3, 4]


def test_planted_window_off_by_one_fails_the_pins(monkeypatch):
    # a window one token too short (the query's own row dropped) frees a block the last query reads
    real = rc.ring_positions_after

    def short_window(n, S, R):
        return real(n, S, max(R - 1, 1)) if R > 1 else real(n, S, R)

    monkeypatch.setattr(rc, "ring_positions_after", short_window)
    with pytest.raises(AssertionError):
        test_dead_blocks_never_hold_a_visible_token_and_only_grow(2, 14, 4)
