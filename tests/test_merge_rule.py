"""The backward's corner-merge rule, restated on the host and checked on
random groups: the kernel's merge must keep every row's total coefficient.

Before the scatter, a point group's samples merge: whole cells (the same
cell offset and level width), or every shared corner (cells on the same level,
W >= 3, that coincide or touch). For each shared corner row, every earlier
holder's original coefficient is added to the last holder, and the earlier
holders skip the row.  This file restates that rule (nine cell offsets, both
corners inside the level) and checks, over random groups with narrow levels,
out-of-level cells and chains, that the rows added and their sums are those
of the unmerged scatter, and that each row is added once.  It also shows the
two ways the rule breaks: without the diagonal offsets, or without the width
guard.
"""
import random

import pytest

MD = 7
CORNERS = [(0, 0), (0, 1), (1, 0), (1, 1)]


def setup(x0, y0, W, H, start):
    wmd = W * MD
    o = start * MD + y0 * wmd + x0 * MD
    mask = sum(1 << k for k, (dy, dx) in enumerate(CORNERS) if 0 <= x0 + dx < W and 0 <= y0 + dy < H)
    return o, wmd, mask


def merge(samples, cells_only=False, diagonals=True, width_guard=True):
    out = []
    for c, (o, wmd, mask, coef) in enumerate(samples):
        mc, smask = list(coef), mask
        for jj, (o2, w2, m2, c2) in enumerate(samples):
            if jj == c or w2 != wmd:
                continue
            pairs = {0: [(0, 0), (1, 1), (2, 2), (3, 3)]}
            if not cells_only:
                if width_guard and wmd < 3 * MD:
                    continue
                pairs.update({MD: [(1, 0), (3, 2)], -MD: [(0, 1), (2, 3)], wmd: [(2, 0), (3, 1)],
                              -wmd: [(0, 2), (1, 3)]})
            if diagonals and not cells_only:
                pairs.update({wmd + MD: [(3, 0)], wmd - MD: [(2, 1)], MD - wmd: [(1, 2)], -MD - wmd: [(0, 3)]})
            for k, k2 in pairs.get(o2 - o, []):
                if (mask >> k) & 1 and (m2 >> k2) & 1:
                    if jj < c:
                        mc[k] += c2[k2]
                    else:
                        smask &= ~(1 << k)
        out.append((mc, smask))
    return out


def failures(trials, **rule):
    rng = random.Random(1)
    bad = 0
    for _ in range(trials):
        levels = [(rng.randint(1, 5), rng.randint(1, 5)) for _ in range(2)]
        starts = [0, levels[0][0] * levels[0][1]]
        samples = []
        for _ in range(4):
            l = rng.randrange(2)
            W, H = levels[l]
            o, wmd, mask = setup(rng.randint(-2, W), rng.randint(-2, H), W, H, starts[l])
            samples.append((o, wmd, mask, [rng.random() for _ in range(4)]))
        want, got, adds = {}, {}, {}
        for o, wmd, mask, coef in samples:
            for k, d in enumerate([0, MD, wmd, wmd + MD]):
                if (mask >> k) & 1:
                    want[o + d] = want.get(o + d, 0.0) + coef[k]
        for (o, wmd, mask, _), (mc, smask) in zip(samples, merge(samples, **rule)):
            assert smask & ~mask == 0
            for k, d in enumerate([0, MD, wmd, wmd + MD]):
                if (smask >> k) & 1:
                    got[o + d] = got.get(o + d, 0.0) + mc[k]
                    adds[o + d] = adds.get(o + d, 0) + 1
        ok = set(got) == set(want) and all(abs(got[r] - want[r]) < 1e-9 for r in want)
        if all(W >= 3 for W, _ in levels) and not rule.get("cells_only"):
            ok = ok and all(v == 1 for v in adds.values())
        bad += not ok
    return bad


@pytest.mark.parametrize("cells_only", [False, True])
def test_merge_keeps_every_row_sum(cells_only):
    assert failures(30000, cells_only=cells_only) == 0


@pytest.mark.parametrize("rule", [dict(diagonals=False), dict(width_guard=False)])
def test_incomplete_rules_lose_coefficients(rule):
    assert failures(30000, **rule) > 0
