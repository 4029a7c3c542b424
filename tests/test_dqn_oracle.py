"""Pins of the DQN-collection oracle (oracle/dqn.c) against things other than
itself: a dueling network whose weights select input components, so that Q is
a closed form of the state (with and without bf16 operand rounding); the LCG
recurrence written out for the exploration draws; the PPO oracle's separately
pinned environment under the same actions; and the TD error's closed form."""
import math

import numpy as np
import pytest

from oracle import dqn
from oracle import oracle as orc
from rl_experience_collection_gb300 import workloads as wl

SD, NA, H, S = wl.STATE_DIM, wl.N_ACTIONS, wl.DQN_H, wl.DQN_S


@pytest.fixture(scope="module", autouse=True)
def _built():
    dqn.build()


def _selector_net():
    """W1 row j picks x[j mod 54]; W2 = I; the value stream averages h2[0..127]
    (+0.25); the advantage stream's row a picks h2[128 + a] (+0.01 a)."""
    parts = {}
    W1 = np.zeros((H, SD), np.float32)
    W1[np.arange(H), np.arange(H) % SD] = 1.0
    Wv1 = np.zeros((S, H), np.float32)
    Wv1[np.arange(S), np.arange(S)] = 1.0
    Wa1 = np.zeros((S, H), np.float32)
    Wa1[np.arange(S), S + np.arange(S)] = 1.0
    Wa2 = np.zeros((NA, S), np.float32)
    Wa2[np.arange(NA), np.arange(NA)] = 1.0
    parts = [W1, np.zeros(H), np.eye(H), np.zeros(H), Wv1, np.zeros(S), np.full((1, S), 1.0 / S), [0.25],
             Wa1, np.zeros(S), Wa2, 0.01 * np.arange(NA)]
    return np.concatenate([np.asarray(p, np.float32).ravel() for p in parts])


def _bf16(v):
    f = np.asarray(v, np.float32).copy()
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64)


def _leaky(v):
    v = np.asarray(v, np.float64)
    return np.where(v < 0, 0.01 * v, v)


def _closed_form(x, rnd):
    h1 = _leaky(rnd(x)[np.arange(H) % SD])
    h2 = _leaky(rnd(h1))
    r2 = rnd(h2)
    hv, ha = _leaky(r2[:S]), _leaky(r2[S:])
    V = np.sum(rnd(hv)) * (1.0 / S) + np.float64(np.float32(0.25))
    A = rnd(ha)[:NA] + (0.01 * np.arange(NA)).astype(np.float32).astype(np.float64)   # float32 biases
    return V, A, V + (A - A.mean())


@pytest.mark.parametrize("quant", ["fp32", "bf16"])
def test_dueling_net_closed_form(quant):
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    cfg = orc.make_cfg(w, quant)
    net = _selector_net()
    assert net.size == dqn.net_count(cfg)
    rnd = _bf16 if quant == "bf16" else (lambda v: np.asarray(v, np.float64))
    rng = np.random.default_rng(1)
    for _ in range(20):
        x = rng.standard_normal(SD) * 3.0
        V, A = dqn.q_parts(net, cfg, x)
        V0, A0, Q0 = _closed_form(x, rnd)
        assert abs(V - V0) <= 1e-12 * max(1, abs(V0))
        np.testing.assert_allclose(A, A0, rtol=1e-12, atol=1e-12)
        q = dqn.q_values(net, cfg, x)
        np.testing.assert_allclose(q, Q0, rtol=1e-12, atol=1e-12)
        assert abs(q.mean() - V0) <= 1e-12 * max(1, abs(V0))       # mean over actions of Q is V


def _lcg(s):
    return (s * 1664525 + 1013904223) & 0xFFFFFFFF


def test_exploration_draws_follow_the_lcg():
    """epsilon = 1: every action is ((s2 >> 8) * 45) >> 24 with s2 the second of
    the step's two LCG states; epsilon = 0: the first argmax of the online Q;
    in between, exploration exactly where u1 = (s1 >> 8) / 2^24 < epsilon."""
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    inp = wl.generate(w, n_episodes=4, horizon=60)
    W = wl.dqn_weights(3, 0.05)
    cfg = orc.make_cfg(w)
    net = dqn.net_count(cfg)
    for eps in (1.0, 0.0, 0.37):
        out = dqn.rollout(w, inp, W, np.arange(4), eps, horizon=60)
        for n in range(4):
            s = int(inp.seeds[n])
            for t in range(60):
                s = _lcg(s)
                u1 = (s >> 8) / 2.0 ** 24
                s = _lcg(s)
                a_rand = ((s >> 8) * 45) >> 24
                assert a_rand == math.floor(((s >> 8) / 2.0 ** 24) * 45)
                q = dqn.q_values(W[:net], cfg, out["states"][n, t].astype(np.float64))
                want = a_rand if u1 < np.float32(eps) else int(np.argmax(q))
                assert out["actions"][n, t] == want, (eps, n, t)
                assert out["q"][n, t] == np.float32(q[want])


def test_environment_is_the_ppo_collectors():
    """Driven by the same actions, the DQN oracle's states, rewards and dones equal
    the PPO oracle's (whose environment is pinned on its own), with the DQN
    curiosity block in the PPO weights."""
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    inp = wl.generate(w, n_episodes=5, horizon=80)
    W = wl.dqn_weights(4, 0.05)
    cfg = orc.make_cfg(w)
    net = dqn.net_count(cfg)
    out = dqn.rollout(w, inp, W, np.arange(5), 0.3, horizon=80)
    ppo_w = inp.weights.copy()
    ppo_w[-wl.dqn_cur_params():] = W[2 * net:]
    inp2 = wl.Inputs(inp.features, inp.starts, inp.seeds, ppo_w)
    ref = orc.rollout(w, inp2, np.arange(5), horizon=80, gpu_actions=out["actions"], act_band=np.inf)
    assert ref["stats"]["action_mismatches"] == 0
    np.testing.assert_array_equal(ref["actions"], out["actions"])
    for k in ("states", "rewards", "dones"):
        np.testing.assert_array_equal(ref[k], out[k], err_msg=k)
    # next_states: the following row where the episode goes on
    cont = out["dones"][:, :-1] == 0
    np.testing.assert_array_equal(out["next_states"][:, :-1][cont], out["states"][:, 1:][cont])
    assert out["dones"].sum() > 0


def test_td_error_closed_form():
    """With the selector net as the target, td = |r + gamma max_a Q_t(x') (1 - d) - q|
    with Q_t in closed form; gamma = 0 leaves |r - q|."""
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    inp = wl.generate(w, n_episodes=3, horizon=50)
    cfg = orc.make_cfg(w, "fp32")
    W = wl.dqn_weights(5, 0.05)
    net = dqn.net_count(cfg)
    W[net:2 * net] = _selector_net()
    for gamma in (0.0, 0.9):
        out = dqn.rollout(w, inp, W, np.arange(3), 0.2, quant="fp32", horizon=50, gamma=gamma)
        for n in range(3):
            for t in range(50):
                _, _, qt = _closed_form(out["next_states"][n, t].astype(np.float64), lambda v: np.asarray(v, np.float64))
                r, q, d = float(out["rewards"][n, t]), float(out["q"][n, t]), out["dones"][n, t]
                want = abs(r + gamma * qt.max() * (1 - d) - q)
                # the oracle forms td from unrounded r and q; the outputs are float32
                assert abs(out["td"][n, t] - want) <= 1e-6 * max(1.0, abs(want)), (gamma, n, t)


@pytest.mark.parametrize("quant", ["fp32", "bf16"])
def test_biases_and_stream_heads_closed_form(quant):
    """W1 = 0 and W2 = I with random biases (half of them negative, so that the
    LeakyReLU slope shows in every layer), selector stream inputs, and random
    stream heads Wv2 [1 x 128], Wa2 [45 x 128]: every bias enters its own layer,
    and the heads are the stated [out, in] products (operands rounded once in
    bf16 mode, biases not)."""
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    cfg = orc.make_cfg(w, quant)
    rng = np.random.default_rng(7)
    f32 = lambda a: np.asarray(a, np.float32)
    b1, b2 = f32(rng.standard_normal(H)), f32(rng.standard_normal(H))
    bv1, ba1 = f32(rng.standard_normal(S)), f32(rng.standard_normal(S))
    Wv2, bv2 = f32(rng.standard_normal((1, S)) * 0.1), f32([0.3])
    Wa2, ba2 = f32(rng.standard_normal((NA, S)) * 0.1), f32(rng.standard_normal(NA) * 0.1)
    Wv1 = np.zeros((S, H), np.float32)
    Wv1[np.arange(S), np.arange(S)] = 1.0
    Wa1 = np.zeros((S, H), np.float32)
    Wa1[np.arange(S), S + np.arange(S)] = 1.0
    parts = [np.zeros((H, SD)), b1, np.eye(H), b2, Wv1, bv1, Wv2, bv2, Wa1, ba1, Wa2, ba2]
    net = np.concatenate([f32(p).ravel() for p in parts])
    assert net.size == dqn.net_count(cfg)
    rnd = _bf16 if quant == "bf16" else (lambda v: np.asarray(v, np.float64))
    d = lambda a: np.asarray(a, np.float64)
    h1 = _leaky(d(b1))                                   # W1 = 0: the state does not matter
    h2 = _leaky(rnd(h1) + d(b2))
    hv = _leaky(rnd(h2)[:S] + d(bv1))
    ha = _leaky(rnd(h2)[S:] + d(ba1))
    V0 = float(rnd(Wv2.ravel()) @ rnd(hv)) + float(bv2[0])
    A0 = rnd(Wa2.ravel()).reshape(NA, S) @ rnd(ha) + d(ba2)
    assert (b1 < 0).any() and (bv1 < 0).any() and (ba1 < 0).any()
    for x in (np.zeros(SD), rng.standard_normal(SD)):
        V, A = dqn.q_parts(net, cfg, x)
        assert abs(V - V0) <= 1e-12 * max(1.0, abs(V0))
        np.testing.assert_allclose(A, A0, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(dqn.q_values(net, cfg, x), V0 + (A0 - A0.mean()), rtol=1e-12, atol=1e-12)


def test_recycling_bars_follow_the_lcg():
    """Episode recycling with a done on every step (a one-bar time barrier) and
    epsilon = 1: each step draws u1, then the random action from the second LCG
    state, then (before the last step) the next bar ((s3 >> 8) * R) >> 24 with
    R = n_bars - L + t + 1 from the third; every state row reads its own bar and
    every next state the bar after it."""
    import dataclasses
    w = dataclasses.replace(wl.DQN_WORKLOADS["dqn_tiny_bf16"], max_hold=1)
    L = 40
    inp = wl.generate(w, n_episodes=3, horizon=L)
    W = wl.dqn_weights(5, 0.05)
    nb = inp.features.shape[0]
    out = dqn.rollout(w, inp, W, np.arange(3), 1.0, horizon=L, recycle=True)
    assert (out["dones"] == 1).all()
    for n in range(3):
        s = int(inp.seeds[n])
        bar = int(inp.starts[n])
        for t in range(L):
            assert out["bars"][n, t] == bar, (n, t)
            np.testing.assert_array_equal(out["states"][n, t, :51], inp.features[bar])
            np.testing.assert_array_equal(out["next_states"][n, t, :51], inp.features[bar + 1])
            s = _lcg(s)
            s = _lcg(s)
            assert out["actions"][n, t] == ((s >> 8) * 45) >> 24, (n, t)
            if t < L - 1:
                s = _lcg(s)
                R = nb - L + t + 1
                bar = ((s >> 8) * R) >> 24
                assert 0 <= bar and bar + (L - 1 - t) <= nb - 1
        # the portfolio restarts with every step: V = 1, e = 0
        assert (out["states"][n, :, 51] == 1.0).all() and (out["states"][n, :, 52] == 0.0).all()


def test_recycling_off_is_the_default_and_on_keeps_the_rules():
    """Without the option the bars are start + t and nothing else changes; with it,
    a step after a done starts at a bar in [0, n_bars - L + t], every other step
    at the next bar, and the states read those bars."""
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    L = 120
    inp = wl.generate(w, n_episodes=6, horizon=L)
    W = wl.dqn_weights(6, 0.05)
    a = dqn.rollout(w, inp, W, np.arange(6), 0.3, horizon=L)
    b = dqn.rollout(w, inp, W, np.arange(6), 0.3, horizon=L, recycle=False)
    for k in ("states", "next_states", "actions", "rewards", "dones", "q", "td", "bars"):
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
    np.testing.assert_array_equal(a["bars"], inp.starts[:6, None] + np.arange(L)[None, :])
    r = dqn.rollout(w, inp, W, np.arange(6), 0.3, horizon=L, recycle=True)
    nb = inp.features.shape[0]
    jumps = 0
    for n in range(6):
        for t in range(L - 1):
            if r["dones"][n, t]:
                assert 0 <= r["bars"][n, t + 1] <= nb - L + t
                jumps += r["bars"][n, t + 1] != r["bars"][n, t] + 1
            else:
                assert r["bars"][n, t + 1] == r["bars"][n, t] + 1
        np.testing.assert_array_equal(r["states"][n, :, :51], inp.features[r["bars"][n]])
        np.testing.assert_array_equal(r["next_states"][n, :, :51], inp.features[r["bars"][n] + 1])
    assert r["dones"].sum() > 0 and jumps > 0
    # up to the first done the two runs agree
    for n in range(6):
        d = np.flatnonzero(r["dones"][n])
        t0 = int(d[0]) + 1 if d.size else L
        np.testing.assert_array_equal(r["actions"][n, :t0], a["actions"][n, :t0])
