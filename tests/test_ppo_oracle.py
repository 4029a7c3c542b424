"""Pins of the PPO-update oracle (oracle/ppo.c) against things other than itself:
central finite differences of its own loss (so the backpropagated gradient
is pinned to the loss's definition), the rollout oracle's separately pinned
actor and critic, and closed forms of the clipped surrogate, the global-norm
clipping and the first Adam step."""
import numpy as np
import pytest
from scipy.special import log_softmax

from rl_experience_collection_gb300 import workloads as wl
from oracle import oracle as orc
from oracle import ppo


@pytest.fixture(scope="module")
def setup():
    ppo.build()
    orc.build()
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.generate(w, n_episodes=4, horizon=4)
    return w, inp


def _batch(w, inp, T, seed, ratio_spread=0.3):
    """T synthetic tuples whose old log-probabilities sit near the actor's own,
    so that the ratios straddle the clip range."""
    rng = np.random.default_rng(seed)
    cfg = orc.make_cfg(w, "fp32")
    states = np.zeros((T, 54), dtype=np.float32)
    states[:, :51] = rng.standard_normal((T, 51)).astype(np.float32)
    states[:, 51] = (1.0 + 0.05 * rng.standard_normal(T)).astype(np.float32)
    states[:, 52] = rng.choice([-1.0, -0.5, 0.0, 0.5, 1.0], size=T).astype(np.float32)
    states[:, 53] = np.float32(w.spread)
    actions = rng.integers(0, 45, size=T).astype(np.int32)
    lp = np.array([log_softmax(orc.actor(inp.weights, cfg, states[i].astype(np.float64)))[actions[i]]
                   for i in range(T)])
    logp_old = (lp + ratio_spread * rng.standard_normal(T)).astype(np.float32)
    adv = rng.standard_normal(T).astype(np.float32)
    ret = rng.standard_normal(T).astype(np.float32)
    return ppo.Batch(states, actions, logp_old, adv, ret), lp


def _loss(p, shape, hp, b, rows):
    st, _ = ppo.loss_grad(p, shape, hp, b, rows)
    return st[0] + hp.value_coef * st[1]


def test_gradient_matches_central_differences(setup):
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, _ = _batch(w, inp, 6, seed=1)
    rows = np.arange(6, dtype=np.int32)
    hp = ppo.Hyper(value_coef=0.7)
    p = inp.weights[:n].astype(np.float64)
    _, g = ppo.loss_grad(p, shape, hp, b, rows)
    rng = np.random.default_rng(7)
    # a spread of entries over every layer, plus each layer's last bias
    idx = list(rng.choice(n, size=40, replace=False))
    idx += [18221 - 1, 128 * 54 + 127, n - 1, n - 2]      # actor b3[44], actor b1[127], critic head b, head w
    for i in idx:
        h = 1e-6 * max(1.0, abs(p[i]))
        pp, pm = p.copy(), p.copy()
        pp[i] += h
        pm[i] -= h
        fd = (_loss(pp, shape, hp, b, rows) - _loss(pm, shape, hp, b, rows)) / (2 * h)
        assert abs(fd - g[i]) <= 1e-6 + 1e-4 * abs(g[i]), (i, fd, g[i])


def test_forward_agrees_with_rollout_oracle_and_ratio_one_closed_form(setup):
    """With old log-probs equal to the actor's own (rollout oracle), every ratio is 1:
    the surrogate is -mean(A), nothing is clipped, and the value loss is the mean
    squared error of the rollout oracle's critic."""
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, lp = _batch(w, inp, 10, seed=2, ratio_spread=0.0)
    b.logp = lp.astype(np.float64).astype(np.float32)
    rows = np.arange(10, dtype=np.int32)
    st, _ = ppo.loss_grad(inp.weights[:n].astype(np.float64), shape, ppo.Hyper(), b, rows)
    cfg = orc.make_cfg(w, "fp32")
    v = np.array([orc.critic(inp.weights, cfg, b.states[i].astype(np.float64)) for i in range(10)])
    assert abs(st[0] - (-b.adv.astype(np.float64).mean())) < 1e-6
    assert abs(st[3] - 1.0) < 1e-6 and st[2] == 0.0
    assert abs(st[1] - np.mean((v - b.ret.astype(np.float64)) ** 2)) < 1e-9 * max(1.0, st[1])


def test_clipped_rows_carry_no_policy_gradient(setup):
    """rho > 1+eps with A > 0, or rho < 1-eps with A < 0: the clipped term is the
    smaller and flat in the actor's parameters, so only the critic has a gradient."""
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, lp = _batch(w, inp, 8, seed=3, ratio_spread=0.0)
    sign = np.where(np.arange(8) % 2 == 0, 1.0, -1.0)
    b.adv = (sign * (0.5 + np.abs(b.adv))).astype(np.float32)
    b.logp = (lp - sign * 0.5).astype(np.float32)         # rho = e^{+-0.5}: outside [0.8, 1.2]
    rows = np.arange(8, dtype=np.int32)
    st, g = ppo.loss_grad(inp.weights[:n].astype(np.float64), shape, ppo.Hyper(), b, rows)
    assert st[2] == 1.0
    assert np.all(g[:18221] == 0.0) and np.any(g[18221:] != 0.0)
    # the surrogate is then -(1/B) sum clip(rho) A with clip(rho) = 1 +- eps
    assert abs(st[0] - (-np.mean(np.where(sign > 0, 1.2, 0.8) * b.adv.astype(np.float64)))) < 1e-9


def test_loss_and_gradient_are_means_over_rows(setup):
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, _ = _batch(w, inp, 5, seed=4)
    p = inp.weights[:n].astype(np.float64)
    hp = ppo.Hyper()
    st_all, g_all = ppo.loss_grad(p, shape, hp, b, np.arange(5, dtype=np.int32))
    parts = [ppo.loss_grad(p, shape, hp, b, np.array([i], dtype=np.int32)) for i in range(5)]
    np.testing.assert_allclose(g_all, np.mean([g for _, g in parts], axis=0), rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(st_all, np.mean([s for s, _ in parts], axis=0), rtol=1e-12, atol=1e-15)
    # the critic's gradient scales with value_coef, the actor's does not
    _, g2 = ppo.loss_grad(p, shape, ppo.Hyper(value_coef=2.0), b, np.arange(5, dtype=np.int32))
    np.testing.assert_array_equal(g2[:18221], g_all[:18221])
    np.testing.assert_allclose(g2[18221:], 2.0 * g_all[18221:], rtol=1e-12, atol=1e-18)


def test_kink_margin_finds_a_pre_activation_at_zero(setup):
    """A bias chosen to cancel one unit's sum on one row puts that row at the kink;
    the other rows stay away from it."""
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, _ = _batch(w, inp, 6, seed=8)
    p = inp.weights[:n].astype(np.float64)
    rows = np.arange(6, dtype=np.int32)
    base = ppo.kink_margin(p, shape, b, rows)
    assert np.all(base > 0)
    W1 = p[:54 * 128].reshape(128, 54)
    x = b.states[3].astype(np.float64)
    p[54 * 128 + 5] = -(W1[5] @ x)                     # actor b1[5]: unit 5 of row 3 at exactly 0
    mg = ppo.kink_margin(p, shape, b, rows)
    assert mg[3] < 1e-15
    assert np.all(mg[[0, 1, 2, 4, 5]] > 1e-12)


def test_adam_first_step_and_global_norm_clip_closed_forms():
    rng = np.random.default_rng(5)
    n = 1000
    g0 = rng.standard_normal(n) * np.logspace(-3, 1, n)
    # no clipping: the first bias-corrected step is -lr g / (|g| + eps)
    hp = ppo.Hyper(max_grad_norm=0.0, lr=1e-3, adam_eps=1e-8)
    p, g, m, v = np.zeros(n), g0.copy(), np.zeros(n), np.zeros(n)
    norm = ppo.adam_step(p, g, m, v, 1, hp)
    assert abs(norm - np.sqrt(np.sum(g0 ** 2))) < 1e-9 * norm
    np.testing.assert_allclose(p, -1e-3 * g0 / (np.abs(g0) + 1e-8), rtol=1e-12)
    # clipping to max_norm: the first moment is (1 - beta1) * g * max_norm / (|g| + 1e-6)
    hp = ppo.Hyper(max_grad_norm=0.5)
    p, g, m, v = np.zeros(n), g0.copy(), np.zeros(n), np.zeros(n)
    ppo.adam_step(p, g, m, v, 1, hp)
    scale = 0.5 / (np.sqrt(np.sum(g0 ** 2)) + 1e-6)
    np.testing.assert_allclose(m, 0.1 * g0 * scale, rtol=1e-12)
    np.testing.assert_allclose(v, 0.001 * (g0 * scale) ** 2, rtol=1e-12)
    # a second step with the same gradient: bias correction with t = 2
    p2, m2, v2 = p.copy(), m.copy(), v.copy()
    ppo.adam_step(p2, g0.copy(), m2, v2, 2, hp)
    gs = g0 * scale
    mh = (0.9 * 0.1 * gs + 0.1 * gs) / (1 - 0.9 ** 2)
    vh = (0.999 * 0.001 * gs ** 2 + 0.001 * gs ** 2) / (1 - 0.999 ** 2)
    np.testing.assert_allclose(p2 - p, -3e-4 * mh / (np.sqrt(vh) + 1e-8), rtol=1e-10)
    # weight decay alone (zero gradient): param -= wd * param
    hp = ppo.Hyper(weight_decay=0.01)
    p, m, v = np.ones(n), np.zeros(n), np.zeros(n)
    ppo.adam_step(p, np.zeros(n), m, v, 1, hp)
    np.testing.assert_allclose(p, 0.99, rtol=1e-15)


def test_trainer_update_runs_steps_in_order(setup):
    """Two steps through Trainer.update equal loss_grad + adam_step by hand."""
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, _ = _batch(w, inp, 6, seed=6)
    rows = np.array([5, 0, 3, 1, 4, 2], dtype=np.int32)
    hp = ppo.Hyper()
    tr = ppo.Trainer(inp.weights, w.critic_h)
    st = tr.update(b, rows, n_steps=2, batch=3, hp=hp)
    p = inp.weights[:n].astype(np.float64)
    m, v = np.zeros(n), np.zeros(n)
    for k in range(2):
        s, g = ppo.loss_grad(p, shape, hp, b, rows[3 * k:3 * k + 3])
        norm = ppo.adam_step(p, g, m, v, k + 1, hp)
        np.testing.assert_allclose(st[k, :4], s, rtol=1e-12)
        assert abs(st[k, 4] - norm) <= 1e-12 * norm
    np.testing.assert_array_equal(tr.w[:n], p.astype(np.float32))
    np.testing.assert_array_equal(tr.w[n:], inp.weights[n:])    # curiosity untouched
    assert tr.t.value == 2


# ------------------------------------------------------------------ ReLU-decision replay

def _hidden(p, w, b, rows):
    """The hidden activations of actor and critic, computed here in float64 with
    numpy from the packed layout: [rows, actor hidden | critic hidden]."""
    views = wl.weight_views(np.concatenate([p, np.zeros(wl.n_params(w.critic_h) - p.size)]).astype(np.float64),
                            w.critic_h)
    out = []
    for r in rows:
        x = b.states[r].astype(np.float64)
        parts = []
        for names in (["actor0", "actor1"], [f"critic{i}" for i in range(len(w.critic_h))]):
            h = x
            for nm in names:
                h = np.maximum(views[nm + ".w"] @ h + views[nm + ".b"], 0.0)
                parts.append(h)
        out.append(np.concatenate(parts))
    return np.array(out, dtype=np.float32)


def test_relu_replay_on_own_activations_changes_nothing(setup):
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, _ = _batch(w, inp, 8, seed=21)
    rows = np.arange(8, dtype=np.int32)
    hp = ppo.Hyper()
    p = inp.weights[:n].astype(np.float64)
    st0, g0 = ppo.loss_grad(p, shape, hp, b, rows)
    act = _hidden(p, w, b, rows)
    assert act.shape == (8, 128 + 64 + sum(w.critic_h))
    st1, g1, rep, mis = ppo.loss_grad_replay(p, shape, hp, b, rows, act)
    assert rep == 0 and mis == 0
    # only the float32 rounding of the adopted activation values separates them
    np.testing.assert_allclose(g1, g0, rtol=0, atol=1e-6 * np.abs(g0).max())
    np.testing.assert_allclose(st1, st0, rtol=1e-6)


def test_relu_replay_adopts_a_kink_decision_and_flags_a_far_one(setup):
    w, inp = setup
    shape = ppo.shape_of(w.critic_h)
    n = ppo.trained_count(shape)
    b, _ = _batch(w, inp, 4, seed=22)
    rows = np.arange(4, dtype=np.int32)
    hp = ppo.Hyper()
    p = inp.weights[:n].astype(np.float64)
    # put the pre-activation of critic unit 5 (first layer) exactly at the kink on row 0
    views = wl.weight_views(inp.weights.copy(), w.critic_h)
    c0 = sum(o * i + o for _, (o, i) in wl.layer_shapes(w.critic_h)[:3])      # offset of the critic's first matrix
    W0 = views["critic0.w"].astype(np.float64)
    x0 = b.states[0].astype(np.float64)
    p[c0 + W0.size + 5] = -float(W0[5] @ x0)                                    # its bias
    act = _hidden(p, w, b, rows)
    col = 128 + 64 + 5
    # the path put it on the positive side, by float32 error: a replay
    act_pos = act.copy()
    act_pos[0, col] = np.float32(1e-7)
    _, g_rep, rep, mis = ppo.loss_grad_replay(p, shape, hp, b, rows, act_pos)
    assert mis == 0 and rep >= 1
    # the same activation on the other side, far from the kink: a mismatch
    r1 = 1 if act[1, col] > 0.1 else 2
    act_far = act.copy()
    act_far[r1, col] = 0.0 if act[r1, col] > 0 else 0.5
    _, _, rep2, mis2 = ppo.loss_grad_replay(p, shape, hp, b, rows, act_far)
    assert mis2 >= 1
