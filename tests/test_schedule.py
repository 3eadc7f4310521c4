"""The decode kernel's copy schedule, modelled on the CPU (host logic: which
page each warp handles and in which order copies are issued; no attention
arithmetic). Checks that the schedule cannot deadlock and that the producer
never waits on a stage more than one barrier phase ahead.

The model of one CTA of the persistent decode kernel (4 consumer warps, a
3-stage ring each, 32-lane producer warp):
- the CTA's share [lo, hi) of the flattened (request, KV head, page) list over
  G = min(grid, max(1, T // 8)) CTAs: shares equal in cost, a page costing 1 and
  each (request, KV head) that starts inside a share LAM pages more when the
  kernel takes the polled merge (LAM = 32), none with the counted merge; with
  few (request, KV head) pairs and a long block table the kernel runs half the
  grid (one CTA per SM), and the model follows it; with LAM = 0,
  lo(c) = c * T // G;
- the share is cut into pieces at (request, KV head) boundaries; the consumers
  meet at the end of every piece (a CTA barrier) before any starts the next;
- page f goes to consumer assign(f); each consumer takes its pages in order,
  page k of consumer c in stage k % 3;
- the producer walks the share 32 pages at a time; a page's round is its
  position in the chunk divided by the round size R (4 pages; the earlier
  rule, a page's index among the chunk's pages of its consumer divided by 3,
  equals R = 12). A page is issued
  once its stage's previous use has been consumed, and a round ends when all
  its pages have been issued (the warp reconverges before the next round).
"""
import numpy as np
import pytest

from paged_kv_decode_gb300 import workloads as W

CONS, RING, CHUNK, PAGE, HKV = 4, 3, 32, 16, 8
ROUND_SIZES = (1, 4, 8, 12)  # the shipped round size (4), earlier ones (8, 12) and another measured
LAM = 32  # the kernel's piece cost for batches (polled merge)
POLL_MAX = 24  # the kernel takes the polled merge when grid <= POLL_MAX * batch * KV heads


class ShareMap:
    """The kernel's share map, in the same integer arithmetic: cost C(f) = f + lam * (pairs starting
    in (0, f]); lo(c) = smallest f with C(f) >= c * Ctot // n; cta(f) = the CTA holding f."""

    def __init__(self, seq_lens, grid, lam, hkv=HKV):
        self.pages = [(int(s) + PAGE - 1) // PAGE for s in seq_lens]
        self.hkv, self.lam, self.batch = hkv, lam, len(self.pages)
        self.pref, self.pcp = [0], [0]
        for p in self.pages:
            self.pref.append(self.pref[-1] + p * hkv)
            self.pcp.append(self.pcp[-1] + (hkv if p > 0 else 0))
        self.T = self.pref[-1]
        self.n = min(grid, max(1, self.T // 8))
        self.Ctot = self.T + lam * max(self.pcp[-1] - 1, 0)

    def request_of(self, f):
        lo_b, hi_b = 0, self.batch - 1
        while lo_b < hi_b:
            mid = (lo_b + hi_b + 1) >> 1
            if self.pref[mid] <= f:
                lo_b = mid
            else:
                hi_b = mid - 1
        return lo_b

    def cost(self, f):
        b = self.request_of(f)
        return f + self.lam * (self.pcp[b] + (f - self.pref[b]) // self.pages[b])

    def lo(self, c):
        y = c * self.Ctot // self.n
        if self.lam == 0:
            return y
        lb, hb = 0, self.batch - 1
        while lb < hb:
            mid = (lb + hb + 1) >> 1
            if self.pref[mid] + self.lam * self.pcp[mid] <= y:
                lb = mid
            else:
                hb = mid - 1
        np_ = self.pages[lb]
        if np_ == 0:
            return self.pref[lb]
        key = self.pref[lb] + self.lam * self.pcp[lb]
        h = min((y - key) // (np_ + self.lam), self.hkv - 1)
        return min(y - self.lam * (self.pcp[lb] + h), self.pref[lb] + (h + 1) * np_)

    def cta(self, f):
        return ((self.cost(f) + 1) * self.n + self.Ctot - 1) // self.Ctot - 1


WIDE_MIN_PAGES = 8192  # the kernel's bound for the wide launch shape (one CTA per SM)


def kernel_launch(seq_lens, grid):
    """(grid, piece cost) the kernel uses for this step: few (request, KV head) pairs and a table that can
    hold a long step take the wide shape (half the grid); the polled merge prices boundaries."""
    pairs = len(seq_lens) * HKV
    max_pages = max(1, max((int(s) + PAGE - 1) // PAGE for s in seq_lens))
    if grid > POLL_MAX * pairs and pairs * max_pages >= WIDE_MIN_PAGES:  # (head_dim 128, as modelled here)
        grid //= 2
    return grid, (LAM if grid <= POLL_MAX * pairs else 0)


def shares(seq_lens, grid, lam=None):
    g, klam = kernel_launch(seq_lens, grid)
    if lam is not None:  # a fixed share rule (the deadlock regression keeps the one of its time)
        g, klam = grid, lam
    sm = ShareMap(seq_lens, g, klam)
    pages, pref = sm.pages, sm.pref
    seg_starts = sorted({int(pref[b]) + h * pages[b] for b in range(len(pages)) if pages[b] for h in range(HKV)})
    return [(sm.lo(c), sm.lo(c + 1)) for c in range(sm.n)], seg_starts


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
    if n == 0:  # an empty share (one that falls inside a boundary's cost): nothing to stream
        return True
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


def all_ctas_finish(seq_lens, assign, grid=304, round_pages=CONS * RING, lam=None):
    sh, segs = shares(seq_lens, grid, lam)
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
    # (with the shares of that time: equal page counts)
    assert not all_ctas_finish(MIXES["short_then_long"], assign_piece, round_pages=None, lam=0)
    assert all_ctas_finish(MIXES["short_then_long"], assign_share, round_pages=None, lam=0)



SHARE_MIXES = [[3, 30000, 5, 9000], [0, 700, 0, 33, 1, 2900, 0], list(range(1, 65)), [40000], [1]]


@pytest.mark.parametrize("lam", [0, 8, LAM, 64])
@pytest.mark.parametrize("grid", [7, 64, 304])
def test_share_map_covers_the_list_and_keeps_holders_consecutive(lam, grid):
    # every page belongs to exactly the CTA cta() names; shares tile [0, T) in order; the CTAs holding a
    # (request, KV head) are consecutive and none of them is empty (the merges rely on both); lam 0 gives
    # equal page counts
    rng = np.random.default_rng(grid + lam)
    mixes = SHARE_MIXES + [[int(x) for x in rng.choice([0, 1, 5, 16, 17, 40, 300, 2000, 12000],
                                                        size=int(rng.integers(1, 40)))] for _ in range(12)]
    for lens in mixes:
        if sum(lens) == 0:
            continue
        for hkv in (1, 2, 8):
            sm = ShareMap(lens, grid, lam, hkv)
            L = [sm.lo(c) for c in range(sm.n + 1)]
            assert L[0] == 0 and L[-1] == sm.T and all(L[i] <= L[i + 1] for i in range(sm.n))
            if lam == 0:
                assert L == [c * sm.T // sm.n for c in range(sm.n + 1)]
            for f in range(sm.T):
                c = sm.cta(f)
                assert L[c] <= f < L[c + 1]
            for b, p in enumerate(sm.pages):
                for h in range(hkv if p else 0):
                    fs = sm.pref[b] + h * p
                    for c in range(sm.cta(fs), sm.cta(fs + p - 1) + 1):
                        assert L[c] < L[c + 1] and L[c] < fs + p and L[c + 1] > fs


def test_piece_cost_moves_pages_from_ctas_with_boundaries():
    # at bs16 a share with a (request, KV head) boundary gets fewer pages than one without
    lens = list(W.config_seq_lens(2))
    sm = ShareMap(lens, 304, LAM)
    starts = {sm.pref[b] + h * p for b, p in enumerate(sm.pages) for h in range(HKV)}
    one, two = [], []
    for c in range(sm.n):
        lo, hi = sm.lo(c), sm.lo(c + 1)
        (two if any(lo < x < hi for x in starts) else one).append(hi - lo)
    assert one and two and np.mean(two) + LAM // 2 < np.mean(one)


def new_row_takers(seq_lens, grid):
    """For the fused append: (CTA, consumer warp) pairs that write each (request, KV head)'s new row,
    by the consumer's rule (the warp whose page walk p_first, p_first + 4, ... of a piece that ends at
    the pair's last page reaches that page), and the consumer the producer feeds that page to."""
    bounds, _ = shares(seq_lens, grid)
    pages = [(int(s) + PAGE - 1) // PAGE for s in seq_lens]
    pref = np.concatenate([[0], np.cumsum(np.asarray(pages, dtype=np.int64) * HKV)])
    takers, fed = {}, {}
    for c, (lo, hi) in enumerate(bounds):
        f = lo
        while f < hi:  # the pieces of the share, as the consumers walk them
            b = int(np.searchsorted(pref, f, side="right") - 1)
            np_ = pages[b]
            h = (f - int(pref[b])) // np_
            seg = int(pref[b]) + h * np_
            fend = min(hi, seg + np_)
            p0, p1 = f - seg, fend - seg
            w0 = (f - lo) % CONS
            for w in range(CONS):
                p_first = p0 + (w - w0 + CONS) % CONS
                if p1 == np_ and p_first <= np_ - 1 and (np_ - 1 - p_first) % CONS == 0:
                    assert np_ - 1 in range(p_first, p1, CONS)  # the warp's walk visits the page
                    takers.setdefault((b, h), []).append((c, w))
            if p1 == np_:
                fed[(b, h)] = (c, (seg + np_ - 1 - lo) % CONS)
            f = fend
    return takers, fed, pages


@pytest.mark.parametrize("grid", [304, 152, 8])
def test_each_new_row_has_one_writer_the_consumer_fed_its_page(grid):
    # the consumer-side fused append: exactly one warp of one CTA writes each (request, KV head)'s new
    # row, and it is the consumer the producer hands that page to ((f - lo) mod 4)
    rng = np.random.default_rng(17 + grid)
    mixes = [W.config_seq_lens(2), [40000], [4096], [1] * 64, [0, 16, 17, 0, 33, 1]]
    mixes += [list(rng.integers(0, 3000, size=int(rng.integers(1, 40)))) for _ in range(60)]
    for lens in mixes:
        takers, fed, pages = new_row_takers(lens, grid)
        want = {(b, h) for b, n in enumerate(pages) if n > 0 for h in range(HKV)}
        assert set(takers) == want and set(fed) == want, lens
        for key in want:
            assert takers[key] == [fed[key]], (lens, key, takers[key], fed[key])
