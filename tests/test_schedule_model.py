"""The stream-K work split of the split kernels, stated as a plain Python
model and checked for the properties the kernels rely on: every real K/V tile
of every (sequence, KV head, head chunk) unit is visited by exactly one CTA;
a unit is cut only at a CTA's first or last segment; the CTAs that hold a cut
unit are exactly cta_of_tile(first) .. cta_of_tile(last); and the merge's
rule for the first partial's slot names the slot that CTA wrote.

The model follows the device code (gqa_schedule.cuh, gqa_merge.cuh): per-row
tile counts, a per-unit charge of `cost` virtual tiles ahead of the unit's
first real tile when lengths differ (0 when every non-empty row has the same
tile count, where the aligned CTA count applies), contiguous ranges
start(c) = floor(c*T/P).  No GPU needed."""
import random

import pytest


def cta_start(c, T, P):
    return (c * T) // P if T >= P else min(c, T)


def cta_of_tile(t, T, P):
    return t if T < P else ((t + 1) * P + T - 1) // T - 1


def span(tiles, cost):
    return tiles + cost if tiles > 0 else 0


def plan(lens, Nmax, BN, U, P0, unit_cost):
    tiles = [(max(0, min(L, Nmax)) + BN - 1) // BN for L in lens]
    nz = [t for t in tiles if t > 0]
    uniform = bool(nz) and min(nz) == max(nz)
    P = P0
    if uniform and len(nz) * U <= P:
        P = len(nz) * U * (P // (len(nz) * U))
    cost = 0 if uniform else unit_cost
    return tiles, sum(span(t, cost) * U for t in tiles), P, cost


def segments(c, tiles, T, P, U, cost):
    """The segments CTA c visits, in order (SegmentCursor::next)."""
    if c >= P:
        return []
    pos, end = cta_start(c, T, P), cta_start(c + 1, T, P)
    pre, b, out = 0, 0, []
    while pos < end:
        sp = span(tiles[b], cost)
        while pos >= pre + sp * U:
            pre += sp * U
            b += 1
            sp = span(tiles[b], cost)
        off = pos - pre
        uib, v0 = divmod(off, sp)
        v1 = min(v0 + (end - pos), sp)
        pos += v1 - v0
        if v1 <= cost:
            continue  # only the unit's charge
        out.append(dict(b=b, uib=uib, t0=max(v0 - cost, 0), t1=v1 - cost, tiles=tiles[b],
                        unit_first=pre + uib * sp + cost))
    return out


def cursor_calls(c, tiles, T, P, U, cost):
    """SegmentCursor::next as the device runs it, call by call, with its early
    end (a row start with no more than a unit's charge left in the range
    ends the walk before that row's length is read).  Returns, per call, the
    segment (or None for the call that returns false), the cursor position
    after the call and the lengths read during the call."""
    if c >= P:
        return [(None, 0, 0)]
    pos, end = cta_start(c, T, P), cta_start(c + 1, T, P)
    pre, b = 0, 0
    if pos < end:  # the plan hands the cursor the row that holds its first tile
        while pos >= pre + span(tiles[b], cost) * U:
            pre += span(tiles[b], cost) * U
            b += 1
    tiles_b = tiles[b] if pos < end else 0
    calls = []
    while True:
        reads, seg = 0, None
        while True:
            if pos >= end:
                break
            sp = span(tiles_b, cost)
            stop = False
            while pos >= pre + sp * U:
                if end - pos <= cost:
                    stop = True
                    break
                pre += sp * U
                b += 1
                tiles_b = tiles[b]
                reads += 1
                sp = span(tiles_b, cost)
            if stop:
                break
            uib, v0 = divmod(pos - pre, sp)
            v1 = min(v0 + (end - pos), sp)
            pos += v1 - v0
            if v1 <= cost:
                continue
            seg = dict(b=b, uib=uib, t0=max(v0 - cost, 0), t1=v1 - cost, tiles=tiles_b,
                       unit_first=pre + uib * sp + cost)
            break
        calls.append((seg, end - pos, reads))
        if seg is None:
            return calls


@pytest.mark.parametrize("seed", range(6))
def test_cursor_last_segment_test_and_no_length_read_after_it(seed):
    """The fused step's early arrival: a CTA's segment is its last exactly
    when the range has no more than a unit's charge left after it; the early
    end of the walk gives the same segments as the plain walk; and the call
    that ends the walk reads no length."""
    rng = random.Random(seed)
    for _ in range(60):
        B = rng.choice([1, 2, 5, 16, 40])
        Nmax = rng.choice([128, 1000, 4096])
        lens = [rng.choice([0, 1, 127, 128, 129, rng.randint(0, Nmax)]) for _ in range(B)]
        U, P0 = rng.choice([1, 2, 8]), rng.choice([1, 3, 17, 148])
        tiles, T, P, cost = plan(lens, Nmax, 128, U, P0, 2)
        for c in range(P0):
            calls = cursor_calls(c, tiles, T, P, U, cost)
            segs = [sg for sg, _, _ in calls if sg is not None]
            assert segs == segments(c, tiles, T, P, U, cost)
            assert calls[-1][0] is None and calls[-1][2] == 0, "the closing call read a length"
            for i, (sg, left, _) in enumerate(calls[:-1]):
                assert (left <= cost) == (i == len(calls) - 2), (c, i, left, cost)


def _check(lens, Nmax, BN, U, P0, unit_cost):
    tiles, T, P, cost = plan(lens, Nmax, BN, U, P0, unit_cost)
    owner, segs = {}, {}
    for c in range(P0):
        segs[c] = segments(c, tiles, T, P, U, cost)
        for i, s in enumerate(segs[c]):
            assert 0 <= s["t0"] < s["t1"] <= s["tiles"]
            for t in range(s["t0"], s["t1"]):
                key = (s["b"], s["uib"], t)
                assert key not in owner, f"tile {key} visited twice"
                owner[key] = c
    assert len(owner) == sum(t * U for t in tiles), "a tile was never visited"
    for c, ss in segs.items():
        for i, s in enumerate(ss):
            if s["t0"] == 0 and s["t1"] == s["tiles"]:
                continue  # whole unit: finished in place
            assert i in (0, len(ss) - 1), "a unit cut in the middle of a range"
            c_lo = cta_of_tile(s["unit_first"], T, P)
            c_hi = cta_of_tile(s["unit_first"] + s["tiles"] - 1, T, P)
            holders = sorted({owner[(s["b"], s["uib"], t)] for t in range(s["tiles"])})
            assert holders == list(range(c_lo, c_hi + 1))
            first = [k for k, x in enumerate(segs[c_lo]) if (x["b"], x["uib"]) == (s["b"], s["uib"])][0]
            slot0 = 2 * c_lo if cta_start(c_lo, T, P) >= s["unit_first"] - cost else 2 * c_lo + 1
            assert slot0 == 2 * c_lo + (0 if first == 0 else 1)
            for cc in range(c_lo + 1, c_hi + 1):
                k = [k for k, x in enumerate(segs[cc]) if (x["b"], x["uib"]) == (s["b"], s["uib"])][0]
                assert k == 0, "a later CTA's piece of a cut unit must be its first segment"


@pytest.mark.parametrize("seed", range(6))
def test_schedule_covers_every_tile_once_and_merges_consistently(seed):
    rng = random.Random(seed)
    for _ in range(300):
        B = rng.randint(1, 70)
        Nmax = rng.choice([128, 300, 1000, 4096])
        mode = rng.random()
        if mode < 0.3:
            lens = [Nmax] * B
        elif mode < 0.5:
            lens = [rng.choice([0, Nmax, rng.randint(1, Nmax)]) for _ in range(B)]
        else:
            lens = [rng.randint(0, Nmax) for _ in range(B)]
        _check(lens, Nmax, rng.choice([64, 128]), rng.choice([1, 2, 4, 8, 16]), rng.choice([1, 7, 148, 296]),
               rng.choice([0, 1, 2, 3, 6, 8, 12]))


def test_charge_moves_real_tiles_away_from_ranges_with_many_units():
    """Ragged lengths: a CTA whose range crosses many short sequences gets
    fewer real tiles than one inside a long sequence."""
    lens = [8192] * 4 + [130] * 40
    tiles, T, P, cost = plan(lens, 8192, 128, 8, 148, 2)
    assert cost == 2
    per_cta = [(sum(s["t1"] - s["t0"] for s in segments(c, tiles, T, P, 8, cost)), len(segments(c, tiles, T, P, 8, cost)))
               for c in range(P)]
    many = [t for t, n in per_cta if n >= 4]
    one = [t for t, n in per_cta if n == 1]
    assert many and one and max(many) < min(one)


# ---------------------------------------------------------------- step counter
MASK64 = (1 << 64) - 1


def _arrive_step(word, epoch, P):
    """One CTA's arrival on the fused step's counter word (gqa_merge.cuh,
    arrive_step), as a generator that yields before every access to the
    shared word so that a scheduler can interleave the CTAs at will.
    `word` is a one-element list (the word in L2); returns the count."""
    tagged = epoch << 32
    yield
    old = word[0]                      # atom_add_acq_rel(cnt, 1)
    word[0] = (old + 1) & MASK64
    if (old >> 32) == epoch:
        return (old + 1) & 0xFFFFFFFF
    cur = (old + 1) & MASK64
    tries = 0
    while True:
        if (cur >> 32) == epoch:
            yield
            old = word[0]              # atom_add_acq_rel(cnt, 1)
            word[0] = (old + 1) & MASK64
            assert (old >> 32) == epoch
            return (old + 1) & 0xFFFFFFFF
        assert tries <= P              # the kernel flags a timeout past this bound
        tries += 1
        yield
        seen = word[0]                 # atom_cas_acq_rel(cnt, cur, tagged | 1)
        if seen == cur:
            word[0] = tagged | 1
            return 1
        cur = seen


def _run_step_arrivals(word, epoch, P, rng):
    """All P CTAs of one call arrive in a random interleaving; the one that
    counts P resets the word to (epoch << 32) | 0 (finish_step).  Returns
    the order of arrival (by the atomic add) and the CTAs elected last."""
    gens = {c: _arrive_step(word, epoch, P) for c in range(P)}
    for g in gens.values():
        next(g)
    order, elected = [], []
    while gens:
        c = rng.choice(list(gens))
        try:
            next(gens[c])
        except StopIteration as stop:
            del gens[c]
            order.append(c)
            if stop.value == P:
                elected.append(c)
                word[0] = epoch << 32
    return order, elected


@pytest.mark.parametrize("seed", range(4))
def test_step_counter_stale_words_never_elect_a_wrong_last_cta(seed):
    """Whatever the counter word holds before a call (uncleared memory, a
    count left by a call of another shape or by a call that stopped half way,
    another call's tag), exactly one CTA is elected, and it is the last of
    the grid to count; the word is then ready for the next call (or a graph
    replay of this one, with the same tag)."""
    rng = random.Random(seed)
    for _ in range(400):
        P = rng.choice([1, 2, 3, 7, 148, 296])
        epoch = rng.randint(1, 2 ** 32 - 1)
        stale_tag = rng.choice([0, rng.randint(1, 2 ** 32 - 1), 0xFFFFFFFF])
        if stale_tag == epoch:
            stale_tag ^= 1
        leftover = rng.choice([0, 1, P - 1, P, P + 5, rng.randint(0, 2 ** 32 - 1)])
        word = [rng.choice([(stale_tag << 32) | leftover, rng.getrandbits(64)])]
        if (word[0] >> 32) == epoch:
            word[0] ^= 1 << 32
        for replay in range(2):  # the call, then a replay with the same tag
            order, elected = _run_step_arrivals(word, epoch, P, rng)
            assert sorted(order) == list(range(P))
            assert elected == [order[-1]], (P, hex(word[0]), elected, order[-1])
            assert word[0] == epoch << 32


@pytest.mark.parametrize("P", [2, 7, 148])
def test_step_counter_retry_bound_holds_in_the_worst_interleaving(P):
    """One CTA's swap fails after every other CTA's add into the stale word
    and once more when another CTA installs the tag: it still counts within
    the kernel's bound of P retries, and exactly the last CTA is elected."""
    epoch = 77
    word = [(5 << 32) | 3]
    gens = {c: _arrive_step(word, epoch, P) for c in range(P)}
    for g in gens.values():
        next(g)
    order, elected = [], []

    def step(c):
        try:
            next(gens[c])
        except StopIteration as stop:
            del gens[c]
            order.append(c)
            if stop.value == P:
                elected.append(c)
                word[0] = epoch << 32

    step(0)                            # CTA 0 adds into the stale word
    for c in range(1, P):
        step(c)                        # another stale add ...
        step(0)                        # ... so CTA 0's swap fails
    if P > 1:
        step(P - 1)                    # the last CTA to add saw the word as it is: its swap installs the tag
        assert word[0] == (epoch << 32) | 1
        step(0)                        # CTA 0's swap fails on the tag, then it adds
    while gens:
        step(min(gens))
    assert sorted(order) == list(range(P))
    assert elected == [order[-1]]
    assert word[0] == epoch << 32


def test_step_counter_fixed_offset_is_the_plain_count_without_a_tag():
    """The mistake the tag guards against, on the model: a plain 32-bit count
    that a call of another shape left at k > 0 elects a CTA that is not the
    last (the count reaches P after P - k arrivals)."""
    P, k = 8, 3
    word = k
    counts = []
    for _ in range(P):
        word += 1
        counts.append(word)
    assert counts.index(P) == P - k - 1 != P - 1


# ------------------------------------------- split-item counter, two halves
def _tag_then_arrive(word, epoch):
    """One CTA of a cut projection item (gqa_proj_tc.cuh): tag_unit_counter
    at the start of its range, add_unit_arrival at the end (gqa_merge.cuh),
    yielding before every access to the word so that the CTAs' steps can be
    interleaved at will.  Returns the count its add saw."""
    yield
    old = word[0]                      # volatile read
    if (old >> 32) != epoch:
        yield
        if word[0] == old:             # atomicCAS(cnt, old, epoch << 32)
            word[0] = epoch << 32
    yield                              # ... the CTA's work on the item ...
    yield
    prev = word[0]                     # atomicAdd(cnt, 1)
    word[0] = (prev + 1) & MASK64
    return (prev + 1) & 0xFFFFFFFF


@pytest.mark.parametrize("seed", range(4))
def test_split_item_counter_tagged_early_elects_the_last_arrival(seed):
    """The projection kernel tags a cut item's counter when a CTA starts and
    counts its arrival with one add at the end.  Whatever the word held
    before (uncleared memory, another call's tag and count), every add lands
    on a word with this call's tag, exactly one CTA sees the full count and
    it is the last to add; the merger's reset leaves the word ready for a
    replay with the same tag."""
    rng = random.Random(100 + seed)
    for _ in range(600):
        n = rng.choice([1, 2, 3, 4])
        epoch = rng.randint(1, 2 ** 32 - 1)
        word = [rng.choice([0, rng.getrandbits(64), (rng.randint(0, 2 ** 32 - 1) << 32) | rng.randint(0, 9)])]
        if (word[0] >> 32) == epoch:
            word[0] ^= 1 << 32
        for replay in range(3):
            gens = {c: _tag_then_arrive(word, epoch) for c in range(n)}
            order, elected = [], []
            while gens:
                c = rng.choice(list(gens))
                try:
                    next(gens[c])
                except StopIteration as stop:
                    del gens[c]
                    order.append(c)
                    if stop.value == n:
                        elected.append(c)
                        word[0] = epoch << 32   # the merger's reset
            assert elected == [order[-1]], (n, replay, elected, order)
            assert word[0] == epoch << 32


def test_split_item_counter_untagged_add_miscounts():
    """Without the early tag, an add on a word another call left at (tag, k)
    reaches n after n - k adds: the tag check is what the early half buys."""
    n, k = 3, 1
    word = (7 << 32) | k
    counts = []
    for _ in range(n):
        word += 1
        counts.append(word & 0xFFFFFFFF)
    assert counts.index(n) == n - k - 1 != n - 1
