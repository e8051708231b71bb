"""The split-K decode's stream-K plan, restated on the host, keeps its invariants.

The decode kernel cuts the batch into equal slices of cost, one per block: a
(sequence, KV head) pair of n chunks costs pair_gap + n units, the pair_gap
units before its first chunk holding nothing. Each block then walks its slice:
the pair cut at the slice's end first, then the rest in order. A pair cut across
blocks is merged by whichever block completes its count of pieces. That block
reads one partial slot per piece: slot first_slot in the block of the pair's
first chunk, slot 0 in the later ones.

This file states that bookkeeping in Python, with the kernel's integer
arithmetic, and checks over random batches, grids and gaps that:
  - every chunk of every pair is streamed exactly once;
  - a pair is "whole" exactly when one block holds all of its chunks;
  - the blocks holding a cut pair's pieces are exactly those the merger counts
    (blocks between the first and last chunk's blocks with a non-empty slice);
  - each piece goes to the slot the merge reads;
  - no block uses one partial slot for two cut pieces.
The GPU tests check the kernel's outputs against the oracle; this checks the
plan's reasoning on many more shapes than they can run.
"""
import random

import pytest


def block_of_unit(x, T, nb):
    return ((x + 1) * nb - 1) // T


def slice_begin(c, T, nb):
    return c * T // nb


def plan(nchs, hkv, nb, gap):
    """Pieces of every block: (block, seq, kvh, k0, n, whole, c_first, c_last, first_slot, slot)."""
    pre = [0]
    for n in nchs:
        pre.append(pre[-1] + n + gap)  # cost per KV head
    T = pre[-1] * hkv
    pieces = []
    for b in range(nb):
        ca, cb = b * T // nb, (b + 1) * T // nb
        if ca >= cb:
            continue
        start = next(s for s in range(len(nchs)) if pre[s] * hkv <= ca < pre[s + 1] * hkv)
        end = next(s for s in range(len(nchs)) if pre[s] * hkv <= cb - 1 < pre[s + 1] * hkv)

        def emit(s, kvh, k0, n, pfirst, pstart, slot):
            nch = nchs[s]
            whole = k0 == 0 and n == nch
            c_first = c_last = b
            first_slot = 0
            if not whole:
                c_first = block_of_unit(pfirst, T, nb)
                c_last = block_of_unit(pfirst + nch - 1, T, nb)
                first_slot = 0 if slice_begin(c_first, T, nb) >= pstart else 1
            pieces.append((b, s, kvh, k0, n, whole, c_first, c_last, first_slot, slot))

        stop = cb
        ebase, epl = pre[end] * hkv, nchs[end] + gap
        epb = ebase + ((cb - 1 - ebase) // epl) * epl
        if epb + epl > cb and epb > ca:
            if epb + gap < cb:
                emit(end, (epb - ebase) // epl, 0, cb - (epb + gap), epb + gap, epb, 1)
            stop = epb
        seq, base = start, pre[start] * hkv
        pl = nchs[seq] + gap
        pos = ca
        kvh = (pos - base) // pl
        k0 = max(0, (pos - base) - kvh * pl - gap)
        count = 0
        while pos < stop:
            pstart = base + kvh * pl
            pend = pstart + pl
            piece_end = min(pend, stop)
            n = (piece_end - (pstart + gap)) - k0
            if n > 0:
                emit(seq, kvh, k0, n, pstart + gap, pstart, 0 if count == 0 else 1)
                count += 1
            pos, k0 = piece_end, 0
            if pos == pend:
                if kvh + 1 < hkv:
                    kvh += 1
                elif pos < stop:
                    seq, base, kvh = seq + 1, pend, 0
                    pl = nchs[seq] + gap
    return T, pieces


def check(nchs, hkv, nb, gap):
    T, pieces = plan(nchs, hkv, nb, gap)
    seen = {}
    for (b, s, kvh, k0, n, *_rest) in pieces:
        assert n > 0
        for k in range(k0, k0 + n):
            assert (s, kvh, k) not in seen, ("streamed twice", s, kvh, k)
            seen[(s, kvh, k)] = b
    assert len(seen) == sum(nchs) * hkv, "a chunk was not streamed"
    by_pair = {}
    for p in pieces:
        by_pair.setdefault((p[1], p[2]), []).append(p)
    slots = {}
    for key, ps in by_pair.items():
        if len(ps) == 1:
            assert ps[0][5], ("one piece but not whole", key)
            continue
        assert not any(p[5] for p in ps), ("cut pair marked whole", key)
        assert len({(p[6], p[7], p[8]) for p in ps}) == 1, ("pieces disagree on bookkeeping", key)
        c_first, c_last, first_slot = ps[0][6], ps[0][7], ps[0][8]
        counted = [c for c in range(c_first, c_last + 1)
                   if slice_begin(c + 1, T, nb) > slice_begin(c, T, nb)]
        assert counted == sorted(p[0] for p in ps), ("merge counts other blocks", key)
        for p in ps:
            assert p[9] == (first_slot if p[0] == c_first else 0), ("slot the merge does not read", p)
            slots.setdefault(p[0], []).append(p[9])
    for b, used in slots.items():
        assert len(used) == len(set(used)), ("a partial slot used twice", b, used)


@pytest.mark.parametrize("gap", [0, 1, 2, 3])
def test_plan_invariants_on_random_batches(gap):
    rng = random.Random(1000 + gap)
    for _ in range(300):
        ns = rng.choice([1, 2, 3, 5, 17, 64])
        hkv = rng.choice([1, 2, 8])
        shape = rng.random()
        if shape < 0.3:
            nchs = [rng.randint(1, 3) for _ in range(ns)]
        elif shape < 0.6:
            nchs = [rng.randint(1, 40) for _ in range(ns)]
        else:
            nchs = [rng.choice([1, 1, 2, 17, 300]) for _ in range(ns)]
        nb = rng.choice([1, 2, 3, 7, 64, 232, 296, 1000])
        check(nchs, hkv, nb, gap)


def test_plan_on_the_bench_shapes():
    """qwen_decode_b128-like (32-token chunks of U[100, 1024] contexts, 8 KV
    heads, 296 blocks) and prefix_decode_b64-like (one to seventeen private
    chunks, 232 blocks), at the gaps the library uses."""
    rng = random.Random(7)
    qwen = [(c + 31) // 32 for c in (rng.randint(100, 1024) for _ in range(128))]
    check(qwen, 8, 296, 1)
    prefix = [max(1, (rng.randint(0, 512) + 1 + 31) // 32) for _ in range(64)]
    check(prefix, 8, 232, 2)


def test_gap_moves_chunks_away_from_blocks_crossing_many_pairs():
    """With a gap, a block whose slice crosses many one-chunk pairs streams
    fewer chunks than one inside a long pair."""
    nchs = [1] * 64 + [640]
    _, pieces0 = plan(nchs, 1, 4, 0)
    _, pieces1 = plan(nchs, 1, 4, 1)
    chunks = lambda ps, b: sum(p[4] for p in ps if p[0] == b)
    assert chunks(pieces0, 0) > chunks(pieces1, 0)
    assert chunks(pieces1, 3) > chunks(pieces0, 3)
