"""Host-side model of the decode kernel's work split, checked for the invariants its merge
relies on (no GPU).

The items of all (sequence, KV head) pairs with tokens lie on a cost axis: every such pair
costs w (its boundary) and then one unit per item, so item x of the q-th pair with tokens
sits at cost x + w (q + 1). CTA c takes the items whose cost lies in [T(c), T(c+1)),
T(c) = ceil(c Ct / n). The merge of a pair derives, from the pair alone, which CTAs hold
its items (c_first .. c_last, skipping CTAs whose range holds none of them) and which
partial slot each uses (1 for the last pair of a CTA that began in an earlier pair, else
0). These tests model that arithmetic in plain integers and check it against the ranges."""

import random

import pytest


def ceil_div(a, b):
    return -(-a // b)


def split(items_per_pair, w, n):
    """Per CTA: (first item, one past its last) from a scan like the kernel's."""
    pairs = [(i, k) for i, k in enumerate(items_per_pair) if k > 0]
    ctot = sum(k + w for _, k in pairs)
    tot = sum(k for _, k in pairs)

    def locate(T):
        cost = item = 0
        for _, k in pairs:
            if T < cost + k + w:
                off = T - cost
                return item + (off - w if off > w else 0)
            cost += k + w
            item += k
        return tot

    return [(locate(ceil_div(c * ctot, n)), locate(ceil_div((c + 1) * ctot, n))) for c in range(n)], ctot, tot


def merge_view(pair_first, pair_n, q, w, n, ctot):
    """What the merge of one pair computes: the CTAs holding it and each one's slot."""
    pair_last = pair_first + pair_n - 1
    wq = w * (q + 1)
    cta_at = lambda x: min((x + wq) * n // ctot, n - 1)  # noqa: E731
    c_first, c_last = cta_at(pair_first), cta_at(pair_last)

    def start_in_pair(cc):
        if cc <= c_first:
            return pair_first
        return min(pair_last + 1, max(pair_first, ceil_div(cc * ctot, n) - wq))

    holders = [cc for cc in range(c_first, c_last + 1) if start_in_pair(cc + 1) > start_in_pair(cc)]
    slot = {cc: (1 if cc == c_first and ceil_div(cc * ctot, n) < pair_first + w * q else 0) for cc in holders}
    return holders, slot


def check(items_per_pair, w, n):
    ranges, ctot, tot = split(items_per_pair, w, n)
    # the ranges partition the items in order
    assert ranges[0][0] == 0 and ranges[-1][1] == tot
    for (a0, a1), (b0, b1) in zip(ranges, ranges[1:]):
        assert a0 <= a1 == b0 <= b1
    owner = {}
    for c, (x0, x1) in enumerate(ranges):
        for x in range(x0, x1):
            owner[x] = c
    slots_used = {}
    first = 0
    q = 0
    for k in items_per_pair:
        if k == 0:
            continue
        holders, slot = merge_view(first, k, q, w, n, ctot)
        assert holders == sorted({owner[x] for x in range(first, first + k)})
        if ctot >= n:  # every CTA range covers a cost unit: the span has no empty CTA
            assert holders == list(range(holders[0], holders[-1] + 1))
        for cc in holders:
            x0 = ranges[cc][0]
            # slot 1 exactly when the CTA began in an earlier pair and shares this one
            assert slot[cc] == (1 if x0 < first else 0)
            if len(holders) > 1:
                key = (cc, slot[cc])
                assert key not in slots_used, ("two shared pairs in one slot", key)
                slots_used[key] = q
        first += k
        q += 1
    return ranges


@pytest.mark.parametrize("w", [0, 1, 16, 32, 500])
@pytest.mark.parametrize("n", [1, 3, 152])
def test_split_invariants_on_random_lengths(w, n):
    rng = random.Random(1000 * w + n)
    for _ in range(40):
        hkv = rng.choice([1, 2, 8])
        lens = [rng.choice([0, 1, rng.randint(1, 40), rng.randint(100, 600)]) for _ in range(rng.randint(1, 24))]
        items = [k for k in lens for _ in range(hkv)]
        if sum(items) == 0:
            continue
        check(items, w, n)


def test_boundary_weight_moves_items_away_from_short_pairs():
    """A CTA that covers many short pairs takes fewer items than one inside a long pair."""
    items = [300] * 4 + [3] * 60 + [300] * 4
    r0 = split(items, 0, 16)[0]
    r16 = split(items, 16, 16)[0]
    load0 = [b - a for a, b in r0]
    load16 = [b - a for a, b in r16]
    assert max(load0) - min(load0) <= 1  # the item split is even
    assert min(load16) < max(load16) - 50  # the cost split is not
    check(items, 16, 16)


def test_equal_lengths_with_no_weight_split_evenly():
    ranges = check([256] * 64, 0, 152)
    loads = [b - a for a, b in ranges]
    assert max(loads) - min(loads) <= 1
