"""Pins for the CPU oracle: each checks it against something other than itself
(closed forms, textbook/library routines, brute force, the pages' tables).

Nothing here needs a GPU.
"""
import itertools
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from rl_experience_collection_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ tables

def _golden_rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def test_weight_layout_matches_page_table(oracle_mod):
    rows = _golden_rows("ppo_weight_layout.txt")
    shapes = dict(wl.layer_shapes(wl.CRITIC_STD))
    page = {}
    for net, key, *dims in rows:
        page.setdefault(net, []).append(tuple(int(d) for d in dims))
    ours_actor = []
    for i in range(3):
        o, n_in = shapes[f"actor{i}"]
        ours_actor += [(o, n_in), (o,)]
    ours_critic = []
    for i in range(6):
        o, n_in = shapes[f"critic{i}"]
        ours_critic += [(o, n_in), (o,)]
    assert page["actor"] == ours_actor
    assert page["critic"] == ours_critic
    assert sum(math.prod(s) for s in page["actor"]) == 18221
    assert sum(math.prod(s) for s in page["critic"]) == 364929
    # the oracle's own layout walks the same packed buffer
    cfg = oracle_mod.make_cfg(wl.WORKLOADS["tiny_fp32"])
    assert oracle_mod.lib().oracle_weight_count(cfg) == wl.n_params(wl.CRITIC_STD)
    cfg4 = oracle_mod.make_cfg(wl.WORKLOADS["ceiling_bf16"])
    assert oracle_mod.lib().oracle_weight_count(cfg4) == wl.n_params(wl.CRITIC_WIDE)


def test_output_buffer_sizes_match_page():
    rows = {r[0]: r[1:] for r in _golden_rows("ppo_output_buffers.txt")}
    words = sum(int(rows[k][0]) for k in ("states", "actions", "old_log_probs", "advantages",
                                          "returns", "dones"))
    assert words == int(rows["download_words_per_tuple"][0])
    n, L = int(rows["default_episodes"][0]), int(rows["default_steps"][0])
    assert n * L * words * 4 == int(rows["download_bytes"][0])
    assert (n, L) == (wl.WORKLOADS["default_fp32"].n_episodes, wl.WORKLOADS["default_fp32"].horizon)


# ------------------------------------------------------------------ LCG

A, CINC, M32 = 1664525, 1013904223, 1 << 32


def _affine_pow(n):
    """(a^n, c*(a^n-1)/(a-1)) mod 2^32 by repeated squaring of the affine map."""
    ra, rc = 1, 0
    ba, bc = A, CINC
    while n:
        if n & 1:
            ra, rc = (ba * ra) % M32, (ba * rc + bc) % M32
        ba, bc = (ba * ba) % M32, (ba * bc + bc) % M32
        n >>= 1
    return ra, rc


@pytest.mark.parametrize("seed", [0, 1, 12345, 0xFFFFFFFF])
def test_lcg_matches_jump_ahead_closed_form(oracle_mod, seed):
    s = seed
    for n in range(1, 200):
        s = oracle_mod.lcg_step(s)
        a, c = _affine_pow(n)
        assert s == (a * seed + c) % M32


def test_lcg_low_bits_have_full_period(oracle_mod):
    # Hull-Dobell: c odd and a-1 divisible by 4 => full period 2^32; the low k
    # bits then cycle with period exactly 2^k.  Check k = 16 directly.
    s0 = 7
    s = s0
    seen = set()
    for i in range(1 << 16):
        seen.add(s & 0xFFFF)
        s = oracle_mod.lcg_step(s)
    assert len(seen) == 1 << 16 and (s & 0xFFFF) == (s0 & 0xFFFF)
    assert CINC % 2 == 1 and (A - 1) % 4 == 0


def test_lcg_uniform_is_top_24_bits(oracle_mod):
    us = oracle_mod.lcg_uniforms(0, 3)
    # first three states from s=0 (jump-ahead above) -> u = (s >> 8) / 2^24
    states = [(_affine_pow(n)[1]) for n in (1, 2, 3)]
    assert list(us) == [(s >> 8) / 2.0 ** 24 for s in states]
    assert states == [1013904223, 1196435762, 3519870697]
    u = oracle_mod.lcg_uniforms(99, 200000)
    assert u.min() >= 0.0 and u.max() < 1.0
    # exact in float32 (24 significant bits)
    assert np.all(u.astype(np.float32).astype(np.float64) == u)
    hist = np.histogram(u, bins=64, range=(0, 1))[0]
    chi2 = ((hist - u.size / 64) ** 2 / (u.size / 64)).sum()
    assert chi2 < 120  # 63 dof, p ~ 1e-5


# ------------------------------------------------------------------ operand rounding

def test_bf16_rounding_matches_torch(oracle_mod):
    rng = np.random.default_rng(0)
    xs = np.concatenate([rng.standard_normal(4000) * 10.0 ** rng.integers(-8, 8, 4000),
                         # exact ties: bf16 value + half an ulp
                         (np.arange(1, 200, dtype=np.float32) * 2 ** -7 + 2 ** -8 * 2 ** -7).astype(np.float32),
                         [0.0, -0.0, 1.0, -3.5, 65504.0]]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).to(torch.float32).numpy()
    got = np.array([oracle_mod.round_bf16(float(x)) for x in xs], np.float32)
    assert np.array_equal(got, ref)


def _tf32_reference(x: float) -> float:
    """Nearest value with an 11-bit significand, ties away from zero (exact rationals)."""
    if x == 0.0:
        return x
    fx = Fraction(x)
    e = math.frexp(abs(x))[1]            # |x| in [2^(e-1), 2^e)
    ulp = Fraction(2) ** (e - 11)        # 11 significant bits
    lo = (abs(fx) // ulp) * ulp
    hi = lo + ulp
    pick = hi if (abs(fx) - lo) >= (hi - abs(fx)) else lo
    return float(pick if x > 0 else -pick)


def _tf32_reference_vec(a: np.ndarray) -> np.ndarray:
    """Vectorised form of the reference above (every step is exact in float64)."""
    a = np.asarray(a, np.float64)
    m, e = np.frexp(np.abs(a))
    ulp = np.ldexp(1.0, e - 11)
    lo = np.floor(np.abs(a) / ulp) * ulp
    hi = lo + ulp
    mag = np.where(np.abs(a) - lo >= hi - np.abs(a), hi, lo)
    return np.where(a == 0, a, np.copysign(mag, a))


def test_tf32_rounding_is_nearest_ties_away(oracle_mod):
    rng = np.random.default_rng(1)
    xs = list((rng.standard_normal(3000) * 10.0 ** rng.integers(-6, 6, 3000)).astype(np.float32))
    xs += [np.float32(1 + 2 ** -11), np.float32(-(1 + 2 ** -11)), np.float32(1 + 3 * 2 ** -11)]
    for x in xs:
        assert oracle_mod.round_tf32(float(x)) == np.float32(_tf32_reference(float(x))), x
    np.testing.assert_array_equal(_tf32_reference_vec(np.array(xs, np.float32)),
                                  [_tf32_reference(float(x)) for x in xs])


# ------------------------------------------------------------------ dense layers and MLPs

def _q(a, mode):
    if mode == "fp32":               # unquantised: full double precision
        return np.asarray(a, np.float64)
    a = np.asarray(a, np.float32)
    if mode == "bf16":
        return torch.from_numpy(a.copy()).to(torch.bfloat16).to(torch.float32).numpy().astype(np.float64)
    if mode == "tf32":
        return _tf32_reference_vec(a)
    raise ValueError(mode)


@pytest.mark.parametrize("shape", [(1, 1), (3, 5), (7, 2), (45, 64)])
@pytest.mark.parametrize("relu", [False, True])
def test_dense_matches_numpy(oracle_mod, shape, relu):
    rng = np.random.default_rng(sum(shape))
    W = rng.standard_normal(shape).astype(np.float32)
    b = rng.standard_normal(shape[0]).astype(np.float32)
    x = rng.standard_normal(shape[1])
    ref = W.astype(np.float64) @ x + b
    if relu:
        ref = np.maximum(ref, 0)
    np.testing.assert_allclose(oracle_mod.dense(W, b, x, relu), ref, rtol=1e-13, atol=1e-13)
    # zero weights -> bias; identity weights -> copy
    np.testing.assert_array_equal(oracle_mod.dense(np.zeros_like(W), b, x, False), b.astype(np.float64))
    if shape[0] == shape[1]:
        np.testing.assert_allclose(oracle_mod.dense(np.eye(shape[0], dtype=np.float32), 0 * b, x, False), x)


def _numpy_nets(weights, critic_h, x, a, mode):
    v = wl.weight_views(weights, critic_h)
    xin = _q(x, mode)
    h = xin
    for i in range(3):
        h = _q(v[f"actor{i}.w"], mode) @ h + v[f"actor{i}.b"]
        if i < 2:
            h = _q(np.maximum(h, 0), mode)
    logits = h
    h = xin
    n = len(critic_h) + 1
    for i in range(n):
        h = _q(v[f"critic{i}.w"], mode) @ h + v[f"critic{i}.b"]
        if i < n - 1:
            h = _q(np.maximum(h, 0), mode)
    value = h[0]
    z = np.concatenate([xin, np.eye(wl.N_ACTIONS)[a]])
    z = _q(np.maximum(_q(v["cur0.w"], mode) @ z + v["cur0.b"], 0), mode)
    pred = _q(v["cur1.w"], mode) @ z + v["cur1.b"]
    return logits, value, pred


@pytest.mark.parametrize("mode", ["fp32", "bf16", "tf32"])
@pytest.mark.parametrize("critic_h", [wl.CRITIC_STD, wl.CRITIC_WIDE])
def test_networks_match_numpy_chain(oracle_mod, mode, critic_h):
    rng = np.random.default_rng(5)
    weights = wl.init_weights(rng, critic_h)
    weights[weights.size // 3] += 0.25
    # non-zero biases so a dropped bias would show
    views = wl.weight_views(weights, critic_h)
    for k, arr in views.items():
        if k.endswith(".b"):
            arr[:] = rng.standard_normal(arr.size).astype(np.float32) * 0.1
    w = wl.WORKLOADS["ceiling_bf16" if critic_h == wl.CRITIC_WIDE else "tiny_fp32"]
    cfg = oracle_mod.make_cfg(w, quant=mode)
    for trial in range(3):
        x = rng.standard_normal(wl.STATE_DIM)
        a = int(rng.integers(0, wl.N_ACTIONS))
        logits, value, pred = _numpy_nets(weights, critic_h, x, a, mode)
        np.testing.assert_allclose(oracle_mod.actor(weights, cfg, x), logits, rtol=1e-12, atol=1e-12)
        assert oracle_mod.critic(weights, cfg, x) == pytest.approx(value, rel=1e-12, abs=1e-12)
        np.testing.assert_allclose(oracle_mod.curiosity(weights, cfg, x, a), pred, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ sampler

def test_sampler_chi_squared_against_softmax(oracle_mod):
    from scipy import stats
    rng = np.random.default_rng(3)
    logits = rng.standard_normal(wl.N_ACTIONS) * 1.5
    p = np.exp(logits - logits.max())
    p /= p.sum()
    us = oracle_mod.lcg_uniforms(2024, 1_000_000)
    _, _, cdf = oracle_mod.sample(logits, 0.5)
    acts = np.searchsorted(cdf, us, side="right")           # min{i : u < cdf_i}
    acts = np.minimum(acts, wl.N_ACTIONS - 1)
    # spot-check that the oracle's own draw agrees with the inverse CDF
    for u, a in zip(us[:2000], acts[:2000]):
        assert oracle_mod.sample(logits, float(u))[0] == a
    counts = np.bincount(acts, minlength=wl.N_ACTIONS)
    chi2, pval = stats.chisquare(counts, p * us.size)
    assert pval > 1e-4, (chi2, pval)


def test_sampler_special_cases(oracle_mod):
    from scipy.special import log_softmax
    # equal logits: a = floor(45 u) away from the boundaries
    eq = np.zeros(wl.N_ACTIONS)
    for u in np.linspace(0.001, 0.999, 301):
        a, lp, _ = oracle_mod.sample(eq, float(u))
        if abs(u * 45 - round(u * 45)) > 1e-9:
            assert a == int(math.floor(u * 45))
        assert lp == pytest.approx(-math.log(45), abs=1e-14)
    # one dominant logit always wins
    dom = np.zeros(wl.N_ACTIONS)
    dom[17] = 50.0
    for u in (2.0 ** -24, 0.3, 0.999999):
        assert oracle_mod.sample(dom, u)[0] == 17
    # u = 0 is below every positive cdf value: the first action
    assert oracle_mod.sample(dom, 0.0)[0] == 0
    # log-prob equals the log-softmax; cdf ends at 1
    rng = np.random.default_rng(4)
    l = rng.standard_normal(wl.N_ACTIONS) * 3
    for u in (0.1, 0.5, 0.9):
        a, lp, cdf = oracle_mod.sample(l, u)
        assert lp == pytest.approx(log_softmax(l)[a], abs=1e-12)
        assert cdf[-1] == pytest.approx(1.0, abs=1e-14)
        assert (a == 0 or cdf[a - 1] <= u) and u < cdf[a]
    # u at/above every cdf value falls back to the last action
    assert oracle_mod.sample(l, 1.0)[0] == wl.N_ACTIONS - 1


# ------------------------------------------------------------------ env pieces

def test_action_factorisation_tables(oracle_mod):
    # exposure {-1,-.5,0,.5,1}[a/9]; cost (1 + order + urgency) * base with order=(a%9)/3, urgency=a%3
    expo = [-1.0, -0.5, 0.0, 0.5, 1.0]
    for a in range(45):
        e_idx, rem = divmod(a, 9)
        order, urg = divmod(rem, 3)
        assert oracle_mod.exposure(a) == expo[e_idx]
        assert oracle_mod.tx_rate(a, 1e-4) == pytest.approx((1 + order + urg) * 1e-4, rel=1e-15)
        assert oracle_mod.category(a) == (0 if e_idx <= 1 else 1 if e_idx == 2 else 2)
    assert oracle_mod.tx_rate(0, 1e-4) == pytest.approx(1e-4) and oracle_mod.tx_rate(8, 1e-4) == pytest.approx(5e-4)


def test_window_entropy_brute_force(oracle_mod):
    from scipy.stats import entropy
    for k in range(1, 7):
        for win in itertools.product(range(3), repeat=k):
            counts = np.bincount(win, minlength=3)
            ref = entropy(counts, base=2)
            assert oracle_mod.window_entropy(win) == pytest.approx(ref, abs=1e-12)
    assert oracle_mod.window_entropy([0, 2]) == 1.0                  # (1,1,0): no penalty
    assert oracle_mod.window_entropy([0, 0, 1]) == pytest.approx(0.9182958340544896)  # penalty
    assert oracle_mod.window_entropy([1]) == 0.0


def test_entropy_decisions_are_far_from_threshold():
    # Every histogram of a window of at most 20 actions has H exactly 1 or at
    # least 1e-3 away from it, so a float32 and a float64 evaluation of H < 1
    # agree.
    worst = 1.0
    for n in range(1, 21):
        for c0 in range(n + 1):
            for c1 in range(n + 1 - c0):
                cs = [c for c in (c0, c1, n - c0 - c1) if c]
                h = -sum(c / n * math.log2(c / n) for c in cs)
                if abs(h - 1.0) > 1e-12:
                    worst = min(worst, abs(h - 1.0))
    assert worst > 1e-3


# ------------------------------------------------------------------ GAE closed forms

def _rand_traj(rng, L, p_done):
    r = rng.standard_normal(L)
    v = rng.standard_normal(L)
    d = (rng.random(L) < p_done).astype(np.int32)
    return r, v, d


def test_gae_lambda_zero_is_td_error(oracle_mod):
    rng = np.random.default_rng(6)
    r, v, d = _rand_traj(rng, 50, 0.2)
    vb, g = 0.7, 0.9
    adv, ret = oracle_mod.gae(r, v, d, vb, g, 0.0)
    vn = np.append(v[1:], vb)
    np.testing.assert_allclose(adv, r + g * vn * (1 - d) - v, atol=1e-14)
    np.testing.assert_allclose(ret, adv + v, atol=1e-14)


def test_gae_undiscounted_no_dones_is_return_minus_value(oracle_mod):
    rng = np.random.default_rng(7)
    r, v, _ = _rand_traj(rng, 40, 0.0)
    d = np.zeros(40, np.int32)
    vb = -1.3
    adv, ret = oracle_mod.gae(r, v, d, vb, 1.0, 1.0)
    ref = np.array([r[t:].sum() + vb - v[t] for t in range(40)])
    np.testing.assert_allclose(adv, ref, atol=1e-12)


def test_gae_double_sum_and_segments(oracle_mod):
    rng = np.random.default_rng(8)
    L, g, lam = 60, 0.97, 0.9
    r, v, d = _rand_traj(rng, L, 0.1)
    vb = 0.4
    adv, _ = oracle_mod.gae(r, v, d, vb, g, lam)
    vn = np.append(v[1:], vb)
    delta = r + g * vn * (1 - d) - v
    for t in range(L):
        # A_t = sum_k (g*lam)^k delta_{t+k}, truncated after the first done
        acc, coef = 0.0, 1.0
        for k in range(t, L):
            acc += coef * delta[k]
            if d[k]:
                break
            coef *= g * lam
        assert adv[t] == pytest.approx(acc, abs=1e-12)
    # each segment equals a stand-alone GAE with a zero bootstrap
    ends = np.flatnonzero(d)
    if ends.size:
        e0 = ends[0]
        sub, _ = oracle_mod.gae(r[:e0 + 1], v[:e0 + 1], d[:e0 + 1], 123.0, g, lam)
        np.testing.assert_allclose(adv[:e0 + 1], sub, atol=1e-12)
