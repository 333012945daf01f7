"""Host-side check of the one-launch decode layer's work split (no GPU).

The layer cuts each task list (gate/up: TPE1 tasks per active expert; down:
TPE2 tasks per active expert) into contiguous per-CTA shares of equal
weight, a task of an expert with r segment rows weighing 1 + r.  Each CTA
caches in shared memory the h rows of every expert its down share touches,
in a buffer of `hrows` rows sized on the host as
min(P, ceil(2P / NC) + 1 + 2T); a share that needed more would be refused
on the device (MOE_DEVERR_BAD_METADATA).  These tests restate the share rule
(first task whose weighted start reaches c*W/NC) and check, over many
routings, that the shares tile the task list exactly once and that no down
share reads more h rows than that bound, for the grouped path and for the
one-row-per-pair segments.
"""
import numpy as np
import pytest


def segments(ids, E):
    """Active experts ascending with [lo, hi) sorted-row ranges."""
    counts = np.bincount(np.asarray(ids).ravel(), minlength=E)
    act = np.nonzero(counts)[0]
    hi = np.cumsum(counts[act])
    lo = hi - counts[act]
    return act, lo, hi


def share_start(w, lo, hi, tpe):
    """Index of the first task whose weighted start is >= w (None when no
    expert's weighted span holds w)."""
    for a in range(len(lo)):
        pa = tpe * (a + lo[a])
        pn = tpe * (a + 1 + hi[a])
        if pa <= w < pn:
            cost = 1 + hi[a] - lo[a]
            return a * tpe + -(-(w - pa) // cost)
    return None


def shares(lo, hi, tpe, NC, P):
    A = len(lo)
    W = tpe * (A + P)
    out = []
    for c in range(NC):
        b = share_start(W * c // NC, lo, hi, tpe)
        b = 0 if b is None else b
        e = share_start(W * (c + 1) // NC, lo, hi, tpe) if c + 1 < NC else None
        e = A * tpe if e is None else e
        out.append((b, e))
    return out


def hrows_bound(T, P, NC):
    return min(P, -(-2 * P // NC) + 1 + 2 * T)


def routing(rng, T, E, k, hot):
    ids = np.empty((T, k), np.int64)
    for t in range(T):
        if hot and rng.random() < 0.7:
            pool = rng.permutation(min(E, max(k, 16)))[:k]
        else:
            pool = rng.permutation(E)[:k]
        ids[t] = pool
    return ids


def check_grouped(ids, E, T, k, tpe, NC):
    _, lo, hi = segments(ids, E)
    A, P = len(lo), T * k
    sh = shares(lo, hi, tpe, NC, P)
    # contiguous and covering every task exactly once
    assert sh[0][0] == 0 and sh[-1][1] == A * tpe
    for c in range(NC - 1):
        assert sh[c][1] == sh[c + 1][0]
        assert sh[c][0] <= sh[c][1]
    bound = hrows_bound(T, P, NC)
    worst = 0
    for b, e in sh:
        if e > b:
            nh = hi[(e - 1) // tpe] - lo[b // tpe]
            worst = max(worst, nh)
            assert nh <= bound, (nh, bound, T, k, E, tpe, NC)
    return worst


@pytest.mark.parametrize("NC", [1, 2, 7, 60, 152])
@pytest.mark.parametrize("tpe", [1, 3, 20, 160])
def test_grouped_down_shares_stay_within_the_h_cache(NC, tpe):
    rng = np.random.default_rng(1000 * NC + tpe)
    for trial in range(60):
        T = int(rng.integers(1, 9))
        E = int(rng.choice([8, 16, 64, 512]))
        k = int(rng.integers(1, min(10, E) + 1))
        if T * k > 256:
            continue
        check_grouped(routing(rng, T, E, k, hot=bool(trial % 2)), E, T, k, tpe, NC)


def test_the_bound_is_met_on_a_worst_case_routing():
    """Every token chooses the same k experts (k rows per segment, the
    longest segments there are) on the decode configurations' geometry."""
    for T in range(1, 9):
        k = 10
        ids = np.tile(np.arange(k), (T, 1))
        for NC in (1, 2, 152):
            check_grouped(ids, 512, T, k, 160, NC)


def test_pair_segments_share_rule_tiles_the_list():
    """Pair segments: P one-row segments, every task of equal weight (the
    closed form the kernel uses), contiguous and within the h bound."""
    def share1(w, tpe):
        a3 = 3 * tpe
        ax = w // a3
        return ax * tpe + (w - ax * a3 + 2) // 3

    for T in (1, 2, 4, 8):
        for k in (1, 2, 10):
            P = T * k
            for tpe in (1, 5, 160, 320):
                for NC in (1, 7, 152):
                    W = 3 * tpe * P
                    b = [share1(W * c // NC, tpe) for c in range(NC)] + [P * tpe]
                    assert b[0] == 0 and all(b[c] <= b[c + 1] for c in range(NC))
                    lo, hi = np.arange(P), np.arange(1, P + 1)
                    bound = hrows_bound(T, P, NC)
                    for c in range(NC):
                        if b[c + 1] > b[c]:
                            nh = hi[(b[c + 1] - 1) // tpe] - lo[b[c] // tpe]
                            assert nh <= bound


def test_the_end_terms_of_the_bound_are_needed():
    """The check bites: shares that cut multi-row segments read more h rows
    than their weight alone allows (ceil(P / NC) + 1), which the 2T term of
    the bound covers."""
    rng = np.random.default_rng(7)
    T, E, k, tpe, NC = 8, 64, 6, 20, 152
    P = T * k
    worst = 0
    for _ in range(200):
        worst = max(worst, check_grouped(routing(rng, T, E, k, hot=True), E, T, k, tpe, NC))
    assert worst > -(-P // NC) + 1
    assert worst <= hrows_bound(T, P, NC)
