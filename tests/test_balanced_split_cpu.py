"""The balanced decode's split of the stage line, checked by brute force on CPU.

Both balanced decode paths lay every sequence's stages end to end (a stage is
16 tokens, 32 for the head-grouped kernel on E4M3 caches), cut the line into R
equal ranges (range r = stages [r*S/R, (r+1)*S/R)), and let each range finish
the pieces (sequence parts) it holds. A piece that one range holds whole is
written in place; any other piece leaves one partial per range that meets it.
The head-grouped kernel's merge kernel finds the cut pieces from the lengths
alone, with one rule: every cut piece is the last piece of the range it starts
in, and that range's entry is the sequence holding stage g1(r) - 1 when it
starts in r and runs past g1(r). Contributor r' keeps its partial in slot
(r' * H_kv + kvh) * 2, plus 1 for the first range when the piece does not start
that range (there it is the range's last piece, not its first).

This test enumerates, for random length mixes, the pieces a range walks stage
by stage (as the stream kernel's cursor does) and checks that the rule lists
exactly the cut pieces, with the contributors and slots each contributor used.
"""
import numpy as np
import pytest


def line_prefix(lens, tt):
    stages = [(int(L) + tt - 1) // tt for L in lens]
    return np.concatenate([[0], np.cumsum(stages)]).astype(np.int64)


def range_start(r, S, R):
    return (r * S) // R


def stage_owner(g, S, R):
    """The range holding line stage g: the largest r with range_start(r) <= g."""
    return ((g + 1) * R - 1) // S


def walked_pieces(pre, R):
    """Per range, the (sequence, first stage, end stage) pieces it holds and
    the partial slot half each cut piece used, from a stage-by-stage walk."""
    S = int(pre[-1])
    N = len(pre) - 1
    seq_of = np.searchsorted(pre, np.arange(S), side="right") - 1
    out = {}
    for r in range(R):
        g0, g1 = range_start(r, S, R), range_start(r + 1, S, R)
        pieces = []
        for g in range(g0, g1):
            s = int(seq_of[g])
            assert 0 <= s < N and pre[s] <= g < pre[s + 1]
            if not pieces or pieces[-1][0] != s:
                pieces.append([s, g, g + 1])
            else:
                pieces[-1][2] = g + 1
        out[r] = [(s, a, b, int(pre[s]), int(pre[s + 1]), g0, g1) for s, a, b in pieces]
    return out


def cut_rule(pre, R):
    """The merge kernel's enumeration: per range, the sequence holding stage
    g1 - 1 when it starts in the range and runs past it."""
    S = int(pre[-1])
    N = len(pre) - 1
    found = {}
    for r in range(R):
        g0, g1 = range_start(r, S, R), range_start(r + 1, S, R)
        if g0 >= g1:
            continue
        lo = int(np.searchsorted(pre[:N], g1 - 1, side="right") - 1)  # largest s: pre[s] <= g1 - 1
        if pre[lo] >= g0 and pre[lo + 1] > g1:
            rb = stage_owner(int(pre[lo + 1]) - 1, S, R)  # owner of the piece's last stage
            found[lo] = (r, rb, 0 if pre[lo] == g0 else 1)
    return found


@pytest.mark.parametrize("seed", range(40))
def test_cut_pieces_and_slots(seed):
    rng = np.random.default_rng(seed)
    kind = seed % 4
    if kind == 0:    # ragged batch, many ranges per sequence
        lens = rng.integers(0, 3000, size=rng.integers(1, 12))
    elif kind == 1:  # more ranges than stages
        lens = rng.integers(0, 40, size=rng.integers(1, 6))
    elif kind == 2:  # many short sequences, few ranges
        lens = rng.integers(1, 600, size=rng.integers(50, 300))
    else:            # one long sequence among short ones, zeros mixed in
        lens = np.concatenate([rng.integers(0, 50, size=rng.integers(1, 20)), [32768]])
        rng.shuffle(lens)
    tt = 32 if seed % 2 else 16
    R = int(rng.choice([38, 76, 152, 304]))
    pre = line_prefix(lens, tt)
    walked = walked_pieces(pre, R)
    found = cut_rule(pre, R)

    # every piece a range walked is either whole in that range or cut
    cut = {}
    for r, pieces in walked.items():
        for s, a, b, ps, pe, g0, g1 in pieces:
            if ps >= g0 and pe <= g1:
                assert (a, b) == (ps, pe)   # a whole piece: all of it, in one range
                continue
            # the slot half the stream kernel writes: 0 = the range's first piece
            half = 0 if ps <= g0 else 1
            cut.setdefault(s, []).append((r, half))
    assert set(cut) == set(found), (sorted(cut), sorted(found))
    for s, contributors in cut.items():
        ra, rb, bit = found[s]
        rs = [r for r, _ in contributors]
        # the contributors are exactly the non-empty ranges ra .. rb, in order
        S = int(pre[-1])
        assert rb == max(rs) and ra == min(rs)
        expect = [r for r in range(ra, rb + 1) if range_start(r, S, R) < range_start(r + 1, S, R)]
        assert rs == expect
        # and the slot half each used is the one the merge reads
        for r, half in contributors:
            assert half == (bit if r == ra else 0)
