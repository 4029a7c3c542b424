"""Whole-episode pins for the oracle: crafted weights force known actions so the
portfolio, barrier, diversity, curiosity, reward, reset and GAE steps reduce to
closed forms that numpy evaluates independently.  No GPU needed.
"""
import dataclasses

import numpy as np
import pytest

from rl_experience_collection_gb300 import workloads as wl


def _forced_weights(critic_h, actor_bias=None, actor_fn=None, value=0.5):
    w = np.zeros(wl.n_params(critic_h), np.float32)
    v = wl.weight_views(w, critic_h)
    if actor_bias is not None:
        v["actor2.b"][:] = actor_bias
    if actor_fn is not None:
        actor_fn(v)
    v[f"critic{len(critic_h)}.b"][:] = value       # zero weights -> V(s) = value everywhere
    return w


def _inputs(w, n, L, weights):
    base = wl.generate(w, n_episodes=n, horizon=L)
    return dataclasses.replace(base, weights=weights)


def _gae_double_sum(r, v, d, vb, g, lam):
    L = r.size
    vn = np.append(v[1:], vb)
    delta = r + g * vn * (1 - d) - v
    adv = np.zeros(L)
    for t in range(L):
        acc, coef = 0.0, 1.0
        for k in range(t, L):
            acc += coef * delta[k]
            if d[k]:
                break
            coef *= g * lam
        adv[t] = acc
    return adv


def _curiosity_zero(feat_next, V2, e2, spread):
    xn = np.concatenate([feat_next.astype(np.float64), [V2, e2, spread]])
    return 0.01 * np.mean(xn ** 2)


def test_forced_flat_action(oracle_mod):
    w = wl.WORKLOADS["tiny_fp32"]
    bias = np.zeros(45, np.float32)
    bias[20] = 60.0                              # exposure index 2 = flat
    inp = _inputs(w, 3, 120, _forced_weights(w.critic_h, bias))
    out = oracle_mod.rollout(w, inp, [0, 1, 2], horizon=120)
    assert np.all(out["actions"] == 20)
    assert np.all(out["states"][:, :, 51] == 1.0) and np.all(out["states"][:, :, 52] == 0.0)
    done_at = np.zeros(120, np.int32)
    done_at[w.max_hold - 1::w.max_hold] = 1      # time barrier every K steps
    for i in range(3):
        np.testing.assert_array_equal(out["dones"][i], done_at)
        b = inp.starts[i] + np.arange(120)
        cur = np.array([_curiosity_zero(inp.features[bb + 1], 1.0, 0.0, w.spread) for bb in b])
        np.testing.assert_allclose(out["rewards"][i], -0.01 + cur, rtol=1e-6, atol=1e-9)
        np.testing.assert_allclose(out["values"][i], 0.5)
        adv = _gae_double_sum(out["rewards"][i].astype(np.float64), np.full(120, 0.5), done_at, 0.5,
                              w.gamma, w.lam)
        np.testing.assert_allclose(out["adv"][i], adv, rtol=1e-5, atol=1e-6)
        np.testing.assert_allclose(out["ret"][i], adv + 0.5, rtol=1e-5, atol=1e-6)
        # states carry the market row of each bar
        np.testing.assert_array_equal(out["states"][i, :, :51], inp.features[b])
        assert np.all(out["states"][i, :, 53] == np.float32(w.spread))


@pytest.mark.parametrize("action,expo,rate", [(36, 1.0, 1e-4), (44, 1.0, 5e-4), (0, -1.0, 1e-4),
                                              (13, -0.5, 3e-4)])
def test_forced_constant_action_barriers(oracle_mod, action, expo, rate):
    w = wl.WORKLOADS["reset_heavy_bf16"]          # sigma 5e-3, theta 0.2 %, K = 10
    bias = np.zeros(45, np.float32)
    bias[action] = 60.0
    L = 150
    inp = _inputs(w, 2, L, _forced_weights(w.critic_h, bias, value=-0.25))
    out = oracle_mod.rollout(w, inp, [0, 1], horizon=L, quant="fp32")
    cat = 0 if action // 9 <= 1 else (1 if action // 9 == 2 else 2)
    for i in range(2):
        assert np.all(out["actions"][i] == action)
        V, e, k = 1.0, 0.0, 0
        for t in range(L):
            bar = inp.starts[i] + t
            g = np.exp(np.float64(inp.features[bar + 1, 0]))
            V2 = V * (1 - abs(expo - e) * rate) * (1 + expo * (g - 1))
            k += 1
            lab = 1 if V2 - 1 >= w.barrier else (-1 if V2 - 1 <= -w.barrier else 0)
            done = lab != 0 or k >= w.max_hold
            beta = {1: 0.5, -1: -0.5, 0: 0.0}[lab]
            cur = _curiosity_zero(inp.features[bar + 1], V2, expo, w.spread)
            r = (V2 / V - 1) * (1 + beta) - 0.01 + cur - 1e-3 * abs(expo)
            assert out["states"][i, t, 51] == np.float32(V) and out["states"][i, t, 52] == np.float32(e)
            assert out["dones"][i, t] == int(done), (t, V2)
            assert out["rewards"][i, t] == pytest.approx(r, rel=1e-6, abs=1e-9)
            if done:
                V, e, k = 1.0, 0.0, 0
            else:
                V, e = V2, expo
        # the reset-heavy barriers fire on price, not only on time
        assert out["dones"][i].sum() > L // w.max_hold


def _cycle_actor(v):
    # logits depend only on the held exposure e = x[52]:
    #   e = 0 -> action 36 (long), e = 1 -> action 0 (short), e = -1 -> action 20 (flat)
    v["actor0.w"][0, 52] = 1.0
    v["actor0.w"][1, 52] = -1.0
    v["actor1.w"][0, 0] = 1.0
    v["actor1.w"][1, 1] = 1.0
    v["actor2.w"][0, 0] = 100.0
    v["actor2.w"][20, 1] = 100.0
    v["actor2.w"][36, 0] = -100.0
    v["actor2.w"][36, 1] = -100.0
    v["actor2.b"][36] = 50.0


@pytest.mark.parametrize("quant", ["fp32", "bf16", "tf32"])
def test_cycling_actions_window_costs_and_resets(oracle_mod, quant):
    w = wl.WORKLOADS["tiny_fp32"]
    L = 130
    inp = _inputs(w, 2, L, _forced_weights(w.critic_h, actor_fn=_cycle_actor, value=0.0))
    out = oracle_mod.rollout(w, inp, [0, 1], horizon=L, quant=quant)
    nxt = {0.0: (36, 1.0, 1e-4), 1.0: (0, -1.0, 1e-4), -1.0: (20, 0.0, 3e-4)}
    for i in range(2):
        V, e, k, win = 1.0, 0.0, 0, []
        for t in range(L):
            a, e2, rate = nxt[e]
            assert out["actions"][i, t] == a
            bar = inp.starts[i] + t
            g = np.exp(np.float64(inp.features[bar + 1, 0]))
            V2 = V * (1 - abs(e2 - e) * rate) * (1 + e2 * (g - 1))
            k += 1
            lab = 1 if V2 - 1 >= w.barrier else (-1 if V2 - 1 <= -w.barrier else 0)
            done = lab != 0 or k >= w.max_hold
            win = (win + [0 if a // 9 <= 1 else (1 if a // 9 == 2 else 2)])[-20:]
            cnt = np.bincount(win, minlength=3)
            p = cnt[cnt > 0] / len(win)
            H = -(p * np.log2(p)).sum()
            div = -0.01 if H < 1.0 else 0.0
            beta = {1: 0.5, -1: -0.5, 0: 0.0}[lab]
            cur = _curiosity_zero(inp.features[bar + 1], V2, e2, w.spread)
            r = (V2 / V - 1) * (1 + beta) + div + cur - 1e-3 * abs(e2)
            assert out["dones"][i, t] == int(done)
            assert out["rewards"][i, t] == pytest.approx(r, rel=1e-6, abs=1e-9)
            if done:
                V, e, k, win = 1.0, 0.0, 0, []
            else:
                V, e = V2, e2


def test_bootstrap_uses_pre_reset_next_state(oracle_mod):
    # critic = identity on x[51] (portfolio value) through ReLU layers, so
    # V_boot equals V' of the final step even when that step ends the episode
    w = wl.WORKLOADS["reset_heavy_bf16"]

    def value_of_v(v):
        v["critic0.w"][0, 51] = 1.0
        for j in range(1, 5):
            v[f"critic{j}.w"][0, 0] = 1.0
        v["critic5.w"][0, 0] = 1.0
    bias = np.zeros(45, np.float32)
    bias[36] = 60.0
    weights = _forced_weights(w.critic_h, bias, actor_fn=value_of_v, value=0.0)
    for L in (7, 10, 23):
        inp = _inputs(w, 2, L, weights)
        out = oracle_mod.rollout(w, inp, [0, 1], horizon=L, quant="fp32")
        for i in range(2):
            V, e = float(out["states"][i, -1, 51]), float(out["states"][i, -1, 52])
            g = np.exp(np.float64(inp.features[inp.starts[i] + L, 0]))
            V2 = V * (1 - abs(1.0 - e) * 1e-4) * g
            assert out["vboot"][i] == pytest.approx(V2, rel=1e-6)
            np.testing.assert_allclose(out["values"][i], out["states"][i, :, 51], rtol=1e-6)


def test_replay_accounting(oracle_mod):
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.generate(w, n_episodes=2, horizon=40)
    ref = oracle_mod.rollout(w, inp, [0, 1], horizon=40)
    # the oracle's own decisions replay with no differences
    same = oracle_mod.rollout(w, inp, [0, 1], horizon=40, gpu_actions=ref["actions"], gpu_dones=ref["dones"])
    assert same["stats"]["action_replays"] == 0 and same["stats"]["action_mismatches"] == 0
    assert same["stats"]["done_mismatches"] == 0
    np.testing.assert_array_equal(same["rewards"], ref["rewards"])
    # a planted far-from-boundary difference is a mismatch, and is adopted
    bad = ref["actions"].copy()
    bad[0, 5] = (bad[0, 5] + 22) % 45
    got = oracle_mod.rollout(w, inp, [0, 1], horizon=40, gpu_actions=bad)
    assert got["stats"]["action_mismatches"] >= 1 and got["stats"]["max_action_gap"] > 1e-5
    assert got["actions"][0, 5] == bad[0, 5]
    # a planted done difference far from the barrier is a mismatch
    badd = ref["dones"].copy()
    t0 = int(np.flatnonzero(badd[1] == 0)[0])
    badd[1, t0] = 1
    got = oracle_mod.rollout(w, inp, [0, 1], horizon=40, gpu_dones=badd)
    assert got["stats"]["done_mismatches"] == 1 and got["dones"][1, t0] == 1


def test_real_weights_statistics(oracle_mod):
    # sanity on the generated workload: actions spread over the action space,
    # finite outputs, resets at least every K steps
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.generate(w)
    out = oracle_mod.rollout(w, inp, [0, 1, 2, 3], horizon=100)
    assert len(np.unique(out["actions"])) > 10
    for k in ("logp", "values", "rewards", "adv", "ret"):
        assert np.all(np.isfinite(out[k]))
    assert np.all(out["logp"] <= 0)
    for i in range(4):
        gaps = np.diff(np.flatnonzero(np.r_[1, out["dones"][i]]))
        assert gaps.max() <= w.max_hold
