"""The decode kernel's copy schedule, modelled on the CPU (host logic: which
page each warp handles and in which order copies are issued; no attention
arithmetic). Checks that the schedule cannot deadlock and that the producer
never waits on a stage more than one barrier phase ahead.

The model of one CTA of the persistent decode kernel (4 consumer warps, a
3-stage ring each, 32-lane producer warp):
- the CTA's share [lo, hi) of the flattened (request, KV head, page) list, with
  lo(c) = c * T // G over G = min(grid, max(1, T // 8)) CTAs;
- the share is cut into pieces at (request, KV head) boundaries; the consumers
  meet at the end of every piece (a CTA barrier) before any starts the next;
- page f goes to consumer assign(f); each consumer takes its pages in order,
  page k of consumer c in stage k % 3;
- the producer walks the share 32 pages at a time; a page's round is its
  position in the chunk divided by the round size R (8 pages; the earlier
  rule, a page's index among the chunk's pages of its consumer divided by 3,
  equals R = 12). A page is issued
  once its stage's previous use has been consumed, and a round ends when all
  its pages have been issued (the warp reconverges before the next round).
"""
import numpy as np
import pytest

from paged_kv_decode_gb300 import workloads as W

CONS, RING, CHUNK, PAGE, HKV = 4, 3, 32, 16, 8
ROUND_SIZES = (1, 4, 8, 12)  # the shipped round size (8), the earlier one (12) and others measured


def shares(seq_lens, grid):
    pages = [(int(s) + PAGE - 1) // PAGE for s in seq_lens]
    pref = np.concatenate([[0], np.cumsum([p * HKV for p in pages])]).astype(np.int64)
    T = int(pref[-1])
    G = min(grid, max(1, T // 8))  # shares of at least 8 pages
    seg_starts = sorted({int(pref[b]) + h * pages[b] for b in range(len(pages)) if pages[b] for h in range(HKV)})
    return [(c * T // G, (c + 1) * T // G) for c in range(G)], seg_starts


def piece_index(lo, hi, seg_starts):
    """piece of each page of the share (pieces split at segment starts)"""
    cuts = [s for s in seg_starts if lo < s < hi]
    out, j = [], 0
    for f in range(lo, hi):
        if j < len(cuts) and f >= cuts[j]:
            j += 1
            while j < len(cuts) and f >= cuts[j]:
                j += 1
        out.append(j)
    return out


def assign_share(lo, hi, seg_starts):
    return [(f - lo) % CONS for f in range(lo, hi)]


def assign_piece(lo, hi, seg_starts):
    """the earlier rule: page p0 + i of a piece goes to consumer i % CONS"""
    starts = [lo] + [s for s in seg_starts if lo < s < hi]
    out, j = [], 0
    for f in range(lo, hi):
        while j + 1 < len(starts) and f >= starts[j + 1]:
            j += 1
        out.append((f - starts[j]) % CONS)
    return out


def simulate(lo, hi, seg_starts, assign, round_pages=CONS * RING):
    n = hi - lo
    piece = piece_index(lo, hi, seg_starts)
    cons = assign(lo, hi, seg_starts)
    k, seen = [], [0] * CONS
    for c in cons:
        k.append(seen[c])
        seen[c] += 1
    where = {(cons[i], k[i]): i for i in range(n)}
    rounds = []
    for m in range(0, n, CHUNK):
        per, rnd = [0] * CONS, {}
        for i in range(m, min(m + CHUNK, n)):
            # round_pages None: the earlier per-consumer rule (index among the consumer's pages // RING)
            r = per[cons[i]] // RING if round_pages is None else (i - m) // round_pages
            rnd.setdefault(r, []).append(i)
            per[cons[i]] += 1
        rounds += [rnd[r] for r in sorted(rnd)]
    round_of = {i: r for r, lst in enumerate(rounds) for i in lst}
    # one barrier phase: the stage's previous use was issued in an earlier round
    for i in range(n):
        prev = where.get((cons[i], k[i] - RING))
        assert prev is None or round_of[prev] < round_of[i]
    issued, done = [False] * n, [False] * n
    nxt = [0] * CONS
    mine = [[i for i in range(n) if cons[i] == c] for c in range(CONS)]
    ri, J = 0, 0
    while True:
        progress = False
        while ri < len(rounds):
            complete = True
            for i in rounds[ri]:
                if issued[i]:
                    continue
                prev = where.get((cons[i], k[i] - RING))
                if prev is None or done[prev]:
                    issued[i] = progress = True
                else:
                    complete = False
            if not complete:
                break
            ri += 1
        for c in range(CONS):
            while nxt[c] < len(mine[c]):
                i = mine[c][nxt[c]]
                if piece[i] != J or not issued[i]:
                    break
                done[i] = progress = True
                nxt[c] += 1
        if all(done[i] for i in range(n) if piece[i] == J) and J < piece[-1]:
            J += 1
            progress = True
        if not progress:
            return all(done)


def all_ctas_finish(seq_lens, assign, grid=304, round_pages=CONS * RING):
    sh, segs = shares(seq_lens, grid)
    return all(simulate(lo, hi, segs, assign, round_pages) for lo, hi in sh)


MIXES = {
    "short_then_long": [3, 30000, 5, 9000],
    "long_then_short": [30000, 3, 9000, 5],
    "one_page_runs": [1, 2, 3, 4, 5, 6, 7, 8, 40000],
    "ragged_1_64": list(range(1, 65)),
    "padding_rows": [700, 0, 33, 0, 0, 1, 2900, 0],
    "bs16": list(W.config_seq_lens(2)),
    "cfg_pairs": list(W.config_seq_lens(5)),
    "long_40k": list(W.config_seq_lens(3)),
}


@pytest.mark.parametrize("round_pages", ROUND_SIZES)
@pytest.mark.parametrize("name", sorted(MIXES))
def test_share_relative_schedule_never_deadlocks(name, round_pages):
    assert all_ctas_finish(MIXES[name], assign_share, round_pages=round_pages)


def test_round_rule_by_position_equals_the_per_consumer_rule():
    # under the share-relative assignment, position // 12 in a chunk is the page's index among the
    # chunk's pages of its consumer, divided by 3 (the rule the kernel used before round sizes)
    for pos in range(CHUNK):
        assert pos // (CONS * RING) == (pos // CONS) // RING


@pytest.mark.parametrize("round_pages", ROUND_SIZES)
@pytest.mark.parametrize("grid", [2 * 148, 2 * 152, 64, 7])
def test_share_relative_schedule_random_mixes(grid, round_pages):
    rng = np.random.default_rng(grid)
    for _ in range(6):
        b = int(rng.integers(1, 40))
        lens = rng.choice([1, 5, 16, 17, 40, 300, 2000, 12000], size=b)
        assert all_ctas_finish(lens, assign_share, grid=grid, round_pages=round_pages), list(lens)


@pytest.mark.parametrize("round_pages", [13, 16, 32])
def test_rounds_larger_than_the_ring_break_the_one_phase_rule(round_pages):
    # a round of more than 12 pages would hold a page and its stage's previous use together;
    # the kernel's static_assert keeps round sizes at most 12
    with pytest.raises(AssertionError):
        all_ctas_finish(MIXES["bs16"], assign_share, round_pages=round_pages)


def test_piece_relative_schedule_deadlocks_on_one_page_runs():
    # the rule the share-relative assignment replaced: eight one-page pieces
    # pile onto consumer 0 and the producer's second round waits on consumers
    # that are held at a piece boundary behind it
    assert not all_ctas_finish(MIXES["short_then_long"], assign_piece, round_pages=None)
    assert all_ctas_finish(MIXES["short_then_long"], assign_share, round_pages=None)

