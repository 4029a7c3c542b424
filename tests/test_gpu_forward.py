"""rollout_forward (include/rollout.h): the actor, critic and curiosity
networks on given states, on the tensor cores in the handle's operand format,
against the oracle's networks (mode Q for tf32 / bf16, float32 weights and
exact arithmetic for fp32), element by element, on random and edge states."""
import dataclasses

import numpy as np
import pytest

from rl_experience_collection_gb300 import workloads as wl

from . import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rl_experience_collection_gb300 import build
    build.build()
    from oracle import oracle as orc
    orc.build()


def _states(w, M, seed):
    """Random states of the environment's form, then edge rows: all zero, large
    positive and negative features, portfolio values far from 1, every exposure."""
    rng = np.random.default_rng(seed)
    x = np.zeros((M, wl.STATE_DIM), np.float32)
    x[:, :wl.N_MARKET] = rng.standard_normal((M, wl.N_MARKET)).astype(np.float32)
    x[:, 51] = rng.uniform(0.5, 1.5, M).astype(np.float32)
    x[:, 52] = (0.5 * (rng.integers(0, 5, M) - 2)).astype(np.float32)
    x[:, 53] = np.float32(w.spread)
    x[0] = 0.0
    x[1, :wl.N_MARKET] = 20.0
    x[2, :wl.N_MARKET] = -20.0
    x[3, 51] = 50.0
    x[4, 51] = 0.0
    x[5, 53] = 1.0
    a = rng.integers(0, wl.N_ACTIONS, M).astype(np.int32)
    a[:2] = [0, wl.N_ACTIONS - 1]
    return x, a


def _check(w, weights, x, a, rtol):
    import torch
    from oracle import oracle as orc
    from rl_experience_collection_gb300 import binding
    h = binding.Rollout.for_workload(w, weights)
    lg, v, cp = h.forward(torch.from_numpy(x).cuda(), torch.from_numpy(a).cuda())
    torch.cuda.synchronize()
    assert h.status() == binding.ROLLOUT_OK
    lg, v, cp = lg.cpu().numpy(), v.cpu().numpy(), cp.cpu().numpy()
    cfg = orc.make_cfg(w)
    worst = {"logits": 0.0, "values": 0.0, "cur_pred": 0.0}
    for m in range(x.shape[0]):
        xo = x[m].astype(np.float64)
        ol = orc.actor(weights, cfg, xo)
        ov = orc.critic(weights, cfg, xo)
        oc = orc.curiosity(weights, cfg, xo, int(a[m]))
        worst["logits"] = max(worst["logits"], float(parity.rel_err(lg[m], ol).max()))
        worst["values"] = max(worst["values"], float(parity.rel_err(np.array([v[m]]), np.array([ov])).max()))
        worst["cur_pred"] = max(worst["cur_pred"], float(parity.rel_err(cp[m], oc).max()))
    print(w.name, worst)
    for k, e in worst.items():
        assert e <= rtol, (k, e, rtol)
    h.close()
    return lg, v, cp


@pytest.mark.parametrize("name", ["tiny_fp32", "scaleout_tf32", "reset_heavy_bf16", "ceiling_bf16"])
def test_forward_matches_oracle_networks(name):
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=4, horizon=4)
    x, a = _states(w, 300, seed=3)
    _check(w, inp.weights, x, a, parity.RTOL[w.dtype])
    # the same with nonzero biases everywhere (the workloads' biases are zero)
    wb = inp.weights.copy()
    views = wl.weight_views(wb, w.critic_h)
    rng = np.random.default_rng(4)
    for k, arr in views.items():
        if k.endswith(".b"):
            arr[:] = rng.uniform(-0.5, 0.5, arr.shape).astype(np.float32)
    _check(w, wb, x[:97], a[:97], parity.RTOL[w.dtype])


def test_forward_follows_device_weight_refresh_and_reports_bad_actions():
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["reset_heavy_bf16"]
    inp = wl.generate(w, n_episodes=4, horizon=4)
    x, a = _states(w, 130, seed=5)
    xs, acts = torch.from_numpy(x).cuda(), torch.from_numpy(a).cuda()
    w2 = inp.weights.copy()
    wl.weight_views(w2, w.critic_h)["critic0.w"][:] *= 0.5
    h = binding.Rollout.for_workload(w, inp.weights)
    h.set_weights_device(torch.from_numpy(w2).cuda())
    got = [t.cpu().numpy() for t in h.forward(xs, acts)]
    fresh = binding.Rollout.for_workload(w, w2)
    want = [t.cpu().numpy() for t in fresh.forward(xs, acts)]
    for g_, w_ in zip(got, want):
        np.testing.assert_array_equal(g_, w_)
    bad = acts.clone()
    bad[7] = wl.N_ACTIONS
    h.forward(xs, bad)
    assert h.status() == binding.ROLLOUT_ERR_RANGE
    h.forward(xs, acts)                          # each call starts from a clean status word
    assert h.status() == binding.ROLLOUT_OK
    h.close()
    fresh.close()
