"""Pins of the prioritised-replay oracle (oracle/per.py) against things other
than itself: the generator's published test vector, exact rational arithmetic
on tiny buffers, a chi-squared test of the sampling frequencies against
p_i / total, closed forms of the importance-sampling weights, and the ring,
update and clamp rules written out case by case."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy import stats

from oracle import per

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "splitmix64_seed1234567.txt")


def _filled(prio, dim=3, seed=0):
    rng = np.random.default_rng(seed)
    n = len(prio)
    r = per.Replay(n, dim)
    r.insert(rng.standard_normal((n, dim)).astype(np.float32), rng.standard_normal((n, dim)).astype(np.float32),
             rng.integers(0, 45, n).astype(np.int32), rng.standard_normal(n).astype(np.float32),
             (rng.random(n) < 0.2).astype(np.uint8))
    r.prio[:] = np.asarray(prio, dtype=np.float32)
    return r


def test_splitmix64_matches_published_vector():
    want = [int(x) for x in open(GOLDEN) if x.strip() and not x.startswith("#")]
    assert [per.splitmix64_output(1234567, n) for n in range(5)] == want
    u = [per.uniform(1234567, n) for n in range(5)]
    assert all(0.0 <= x < 1.0 for x in u)
    assert u[0] == (want[0] >> 11) / 2.0 ** 53


def test_sampled_slot_holds_the_target_exactly_on_tiny_buffers():
    """In exact rational arithmetic, slot i is picked iff c_{i-1} <= t < c_i:
    zero-priority slots never, the boundary itself belongs to the next slot."""
    rng = np.random.default_rng(1)
    for trial in range(30):
        n = int(rng.integers(1, 12))
        p = rng.random(n).astype(np.float32) * np.float32(3.0)
        p[rng.random(n) < 0.3] = 0.0
        if not p.any():
            p[0] = 1.0
        r = _filled(p)
        idx, _, _, _ = r.sample(40, 0.4, seed=trial, offset=7)
        P = [Fraction(float(x)) for x in p]
        total = sum(P)
        for k, i in enumerate(idx):
            t = Fraction(per.uniform(trial, 7 + k)) * total
            lo = sum(P[:i])
            # the oracle sums in double: allow only a double rounding of the total
            assert P[i] > 0
            assert lo <= t * (1 + Fraction(1, 2 ** 50)) and t < (lo + P[i]) * (1 + Fraction(1, 2 ** 50))
    # a target exactly on a boundary goes to the next positive slot
    r = _filled([1.0, 0.0, 0.0, 1.0])
    c = r.cumulative()
    assert int(np.searchsorted(c, 1.0, side="right")) == 3


def test_sampling_frequencies_follow_priorities():
    rng = np.random.default_rng(2)
    p = (rng.random(40) ** 3).astype(np.float32)
    p[[3, 17]] = 0.0
    r = _filled(p)
    counts = np.zeros(40)
    n = 0
    for call in range(40):
        idx, _, _, _ = r.sample(2000, 0.4, seed=99, offset=call * 2000)
        counts += np.bincount(idx, minlength=40)
        n += 2000
    assert counts[3] == 0 and counts[17] == 0
    pos = p > 0
    expect = n * p[pos].astype(np.float64) / p.astype(np.float64).sum()
    chi2, pval = stats.chisquare(counts[pos], expect)
    assert pval > 1e-4, (chi2, pval)


def test_importance_weights_closed_forms():
    # equal priorities: every weight is 1
    r = _filled(np.full(10, 0.7, dtype=np.float32))
    _, w, _, _ = r.sample(50, 0.6, seed=3, offset=0)
    np.testing.assert_array_equal(w, np.ones(50, dtype=np.float32))
    # w_k = (p_min_in_batch / p_k)^beta: the N and the total cancel
    p = np.array([1.0, 2.0, 4.0, 8.0], dtype=np.float32)
    r = _filled(p)
    for beta in (0.0, 0.4, 1.0):
        idx, w, _, _ = r.sample(64, beta, seed=4, offset=0)
        pmin = p[idx].min()
        np.testing.assert_allclose(w, (pmin / p[idx]) ** beta, rtol=1e-6)
        assert w.max() == 1.0


def test_insert_wraps_and_takes_the_running_max_priority():
    r = per.Replay(5, 2)
    rows = lambda a, b: np.arange(a, b, dtype=np.float32)[:, None].repeat(2, 1)
    ids = lambda a, b: np.arange(a, b, dtype=np.int32)
    r.insert(rows(0, 3), rows(100, 103), ids(0, 3), ids(0, 3).astype(np.float32), np.zeros(3, np.uint8))
    assert (r.size, r.cursor) == (3, 3)
    np.testing.assert_array_equal(r.prio, [1, 1, 1, 0, 0])
    r.update(np.array([1]), np.array([3.0], np.float32), 1.0, 0.0)           # max priority 3
    r.update(np.array([1]), np.array([0.5], np.float32), 1.0, 0.0)           # max stays 3
    assert r.max_prio == 3.0 and r.prio[1] == 0.5
    r.insert(rows(3, 7), rows(103, 107), ids(3, 7), ids(3, 7).astype(np.float32), np.ones(4, np.uint8))
    assert (r.size, r.cursor) == (5, 2)
    np.testing.assert_array_equal(r.actions, [5, 6, 2, 3, 4])               # 5 and 6 wrapped onto 0 and 1
    np.testing.assert_array_equal(r.prio, [3, 3, 1, 3, 3])
    np.testing.assert_array_equal(r.next_states[:, 0], [105, 106, 102, 103, 104])
    # more than the capacity in one call: the last `capacity` survive, in ring order
    r.insert(rows(10, 22), rows(0, 12), ids(10, 22), ids(10, 22).astype(np.float32), np.zeros(12, np.uint8))
    assert (r.size, r.cursor) == (5, 4)
    np.testing.assert_array_equal(r.actions, [18, 19, 20, 21, 17])             # item j to slot (2 + j) mod 5


def test_update_rules():
    r = _filled(np.ones(6, dtype=np.float32))
    r.update(np.array([0, 1, 2, 0, 9, -1]), np.array([2.0, -0.25, 0.0, 4.0, 1.0, 1.0], np.float32), 0.5, 0.01)
    assert r.range_error
    eps = float(np.float32(0.01))
    assert r.prio[0] == np.float32(2.0 + eps)                          # |4|^0.5 + eps: the later entry wins
    assert r.prio[1] == np.float32(0.5 + eps) and r.prio[2] == np.float32(eps)
    # the running max counts the overwritten value too: max(1, sqrt2+eps, 2+eps)
    assert r.max_prio == np.float32(2.0 + eps)
    # alpha = 0: every priority is 1 + eps, whatever the error (0^0 = 1)
    r.update(np.array([3, 4]), np.array([0.0, 123.0], np.float32), 0.0, 0.01)
    assert r.prio[3] == r.prio[4] == np.float32(1.0 + eps)
    # NaN -> eps; inf (and overflow past float32) -> the max priority before the call
    before = r.max_prio
    r.update(np.array([5, 1, 2]), np.array([np.nan, np.inf, 3e38], np.float32), 2.0, 0.01)
    assert r.prio[5] == np.float32(eps)
    assert r.prio[1] == before and r.prio[2] == before and r.max_prio == before
    # the value is computed in double and rounded once
    r.update(np.array([0]), np.array([0.1], np.float32), 0.6, 1e-6)
    assert r.prio[0] == np.float32(float(np.float32(0.1)) ** float(np.float32(0.6)) + float(np.float32(1e-6)))


def test_zero_total_is_refused_and_replay_is_checked():
    r = _filled(np.zeros(4, dtype=np.float32))
    with pytest.raises(ValueError):
        r.sample(4, 0.4, 0, 0)
    # replay only inside the band, and only to a neighbouring slot
    r = _filled(np.array([1.0, 1.0, 1.0], dtype=np.float32))
    idx, _, margin, _ = r.sample(8, 0.4, 5, 0)
    far = margin > 1e-12
    assert far.all()
    bad = idx.copy()
    bad[0] = (bad[0] + 1) % 3
    idx2, _, _, n = r.sample(8, 0.4, 5, 0, replay=bad)                 # outside the band: ignored
    np.testing.assert_array_equal(idx2, idx)
    assert n == 0


def test_update_equals_the_batch_order_loop():
    """Brute force: the update applied entry by entry, in batch order."""
    rng = np.random.default_rng(9)
    for trial in range(40):
        n = int(rng.integers(1, 30))
        r = _filled(np.ones(n, dtype=np.float32))
        B = int(rng.integers(1, 60))
        idx = rng.integers(-2, n + 2, B)
        td = rng.standard_normal(B).astype(np.float32) * 3
        td[rng.random(B) < 0.1] = np.nan
        td[rng.random(B) < 0.1] = np.inf
        alpha, eps = float(rng.choice([0.0, 0.6, 1.0, 2.0])), float(rng.choice([0.0, 1e-6, 0.01]))
        want = r.prio.copy()
        m = r.max_prio
        snap = m
        for k in range(B):
            i = int(idx[k])
            if not 0 <= i < n:
                continue
            if math.isnan(float(td[k])):
                v = np.float32(eps)
            else:
                with np.errstate(over="ignore"):
                    v = np.float32(abs(float(td[k])) ** float(np.float32(alpha)) + float(np.float32(eps)))
                if math.isinf(v):
                    v = snap
            want[i] = v
            m = max(m, v)
        r.update(idx, td, alpha, eps)
        np.testing.assert_array_equal(r.prio, want)
        assert r.max_prio == m
        assert r.range_error == bool(((idx < 0) | (idx >= n)).any())
