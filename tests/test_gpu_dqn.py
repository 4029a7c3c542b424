"""The DQN experience collector (include/dqn.h) against the oracle (oracle/dqn.c)
on the same seeded inputs.

Tolerances (the collector's bf16 tensor-core contract, as for the PPO path):
  * actions, dones, the market and exposure columns of the states and next
    states: exact.  Where the greedy action differs and the two actions' Q
    values lie within Q_BAND * max(1, max |Q|) (a floating-point decision
    between near-equal values) the oracle adopts the GPU's action and counts a
    replay; dones as in the PPO parity (DONE_BAND);
  * V (state column 51): float32 rounding, 2e-6 relative;
  * rewards: abs 5e-2; q: |g - o| <= 2e-2 max(|o|, 1) (values);
  * td = |r + gamma max Q_t - q|: its error is at most the reward's plus the two
    values': 5e-2 + 2e-2 (2 |q| + |td| + 1).
"""
import numpy as np
import pytest

from rl_experience_collection_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

Q_BAND = 2e-3
DONE_BAND = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rl_experience_collection_gb300 import build
    build.build()
    from oracle import dqn
    dqn.build()


def _run(w, inp, W, N, L, eps, next_states=True, starts=None, recycle=False):
    import torch
    from rl_experience_collection_gb300 import binding
    h = binding.DqnCollector.for_workload(w, W, n_bars=inp.features.shape[0])
    if recycle:
        h.set_recycle(True)
    out = binding.make_dqn_outputs(N, L, next_states=next_states)
    st = inp.starts[:N] if starts is None else starts
    h.run(torch.from_numpy(inp.features).cuda(), torch.from_numpy(np.ascontiguousarray(st)).cuda(),
          torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda(), N, L, w.gamma, eps, out)
    status = h.status()
    h.close()
    return status, {k: v.cpu().numpy() for k, v in out.items()}


def _compare(w, inp, W, g, idx, L, eps, recycle=False, ref_out=None):
    from oracle import dqn
    sel = np.asarray(idx)
    ref = dqn.rollout(w, inp, W, sel, eps, horizon=L, gpu_actions=g["actions"], gpu_dones=g["dones"],
                      q_band=Q_BAND, done_band=DONE_BAND, threads=16, recycle=recycle)
    if ref_out is not None:
        ref_out.update(ref)
    st = ref["stats"]
    assert st["action_mismatches"] == 0 and st["done_mismatches"] == 0, st
    g = {k: v[sel] for k, v in g.items()}
    np.testing.assert_array_equal(g["actions"], ref["actions"])
    np.testing.assert_array_equal(g["dones"], ref["dones"])
    for k in ("states", "next_states"):
        if k not in g:
            continue
        np.testing.assert_array_equal(g[k][..., :51], ref[k][..., :51], err_msg=k)
        np.testing.assert_array_equal(g[k][..., 52:], ref[k][..., 52:], err_msg=k)
        np.testing.assert_allclose(g[k][..., 51], ref[k][..., 51], rtol=2e-6, atol=0, err_msg=k)
    r64 = {k: ref[k].astype(np.float64) for k in ("rewards", "q", "td")}
    print(f"max |d rewards| {np.abs(g['rewards'] - r64['rewards']).max():.3e}  "
          f"max rel d q {(np.abs(g['q'] - r64['q']) / np.maximum(np.abs(r64['q']), 1.0)).max():.3e}  "
          f"max |d td| {np.abs(g['td'] - r64['td']).max():.3e}")
    assert np.abs(g["rewards"] - r64["rewards"]).max() <= 5e-2
    assert (np.abs(g["q"] - r64["q"]) / np.maximum(np.abs(r64["q"]), 1.0)).max() <= 2e-2
    tol = 5e-2 + 2e-2 * (2 * np.abs(r64["q"]) + np.abs(r64["td"]) + 1.0)
    assert (np.abs(g["td"] - r64["td"]) <= tol).all()
    assert (g["td"] >= 0).all()
    return st


@pytest.mark.parametrize("N,L,eps,next_states", [(300, 40, 0.1, True), (129, 25, 0.6, False), (1, 7, 0.0, True),
                                                  (641, 100, 0.1, True), (130, 1, 0.3, True)])
def test_dqn_matches_oracle(N, L, eps, next_states):
    """Several CTAs with a ragged last one; exploration-heavy without the optional
    next states; a single episode acting greedily; 501 target-pass tiles, so that
    every CTA of the target pass takes several (both TMEM region assignments,
    the next tile's layer 1 issued inside the current one) and the last tile is
    ragged; a one-step horizon, where every row is its episode's last step (the
    next state's features come from the feature matrix, never from the next row)."""
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    W = wl.dqn_weights(N, 0.05)
    status, g = _run(w, inp, W, N, L, eps, next_states)
    assert status == binding.ROLLOUT_OK
    st = _compare(w, inp, W, g, np.arange(N), L, eps)
    assert st["action_replays"] <= max(2, N * L // 2000)
    if L > w.max_hold:                       # the time barrier alone ends every episode by then
        assert g["dones"].sum() > 0


@pytest.mark.parametrize("N,L,eps", [(300, 60, 0.1), (129, 200, 0.3), (1, 40, 0.0)])
def test_dqn_recycling_matches_oracle(N, L, eps):
    """Episode recycling: after a done the next step starts at a bar drawn from
    the episode's LCG.  The states' market columns are compared exactly, so every
    recycled bar is checked; the next states of done steps stay the pre-reset
    state at the bar after their own.  Several rollout CTAs with a ragged last
    one; 202 target-pass tiles (several per CTA, rows of one warp spanning
    recycled bars); a single greedy episode."""
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    W = wl.dqn_weights(N + 3, 0.05)
    status, g = _run(w, inp, W, N, L, eps, recycle=True)
    assert status == binding.ROLLOUT_OK
    ref = {}
    st = _compare(w, inp, W, g, np.arange(N), L, eps, recycle=True, ref_out=ref)
    assert st["action_replays"] <= max(2, N * L // 2000)
    nb = inp.features.shape[0]
    bars = ref["bars"]
    plain = inp.starts[:N, None].astype(np.int64) + np.arange(L)[None, :]
    assert (bars >= 0).all() and (bars + (L - np.arange(L))[None, :] <= nb - 1).all()
    if N > 1:
        assert (bars != plain).any()          # some episodes did recycle
        # a recycled step's state holds a fresh portfolio
        d = g["dones"][:, :-1].astype(bool)
        np.testing.assert_array_equal(g["states"][:, 1:, 51][d], 1.0)
        np.testing.assert_array_equal(g["states"][:, 1:, 52][d], 0.0)


def test_recycling_off_again_restores_the_plain_run():
    """set_recycle(False) after a recycling run gives the default outputs again."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    N, L = 140, 50
    inp = wl.generate(w, n_episodes=N, horizon=L)
    W = wl.dqn_weights(11, 0.05)
    _, g0 = _run(w, inp, W, N, L, 0.2)
    h = binding.DqnCollector.for_workload(w, W, n_bars=inp.features.shape[0])
    args = (torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts[:N]).cuda(),
            torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda(), N, L, w.gamma, 0.2)
    outs = []
    for on in (True, False):
        h.set_recycle(on)
        out = binding.make_dqn_outputs(N, L)
        h.run(*args, out)
        assert h.status() == binding.ROLLOUT_OK
        outs.append({k: v.cpu().numpy() for k, v in out.items()})
    h.close()
    assert not np.array_equal(outs[0]["states"], g0["states"])
    for k in g0:
        np.testing.assert_array_equal(outs[1][k], g0[k], err_msg=k)


def test_out_of_range_start_and_determinism():
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    N, L = 140, 20
    inp = wl.generate(w, n_episodes=N, horizon=L)
    W = wl.dqn_weights(7, 0.05)
    starts = inp.starts[:N].copy()
    starts[5] = inp.features.shape[0] - L          # start + L > n_bars - 1
    s1, g1 = _run(w, inp, W, N, L, 0.2, starts=starts)
    assert s1 == binding.ROLLOUT_ERR_RANGE
    for k, v in g1.items():
        assert not v[5].any(), k
    keep = np.setdiff1d(np.arange(N), [5])
    _compare(w, wl.Inputs(inp.features, starts, inp.seeds, inp.weights), W, g1, keep, L, 0.2)
    s2, g2 = _run(w, inp, W, N, L, 0.2, starts=starts)
    for k in g1:
        np.testing.assert_array_equal(g1[k], g2[k], err_msg=k)


def test_argument_validation():
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    inp = wl.generate(w, n_episodes=4, horizon=5)
    W = wl.dqn_weights(1)
    h = binding.DqnCollector.for_workload(w, W, n_bars=inp.features.shape[0])
    out = binding.make_dqn_outputs(4, 5)
    args = (torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts).cuda(),
            torch.from_numpy(inp.seeds.view(np.int32)).cuda(), 4, 5, 0.99)
    for eps in (-0.1, 1.5, float("nan")):
        with pytest.raises(binding.RolloutError):
            h.run(*args, eps, out)
    bad = dict(out)
    bad["td"] = None
    with pytest.raises(binding.RolloutError):
        h.run(*args, 0.1, bad)
    with pytest.raises(ValueError):
        binding.DqnCollector.for_workload(w, W[:-1], n_bars=inp.features.shape[0])
    Wn = W.copy()
    Wn[100] = np.inf
    with pytest.raises(binding.RolloutError):
        h.set_weights(Wn)
    h.close()


def test_full_size_sampled_episodes():
    """The benchmark's launch (16384 episodes x 1000 steps): eight episodes spread
    over the CTAs against the oracle, and properties of every transition."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_reset_heavy_bf16"]
    N, L = w.n_episodes, w.horizon
    inp = wl.generate(w)
    W = wl.dqn_weights(w.seed, 0.05)
    h = binding.DqnCollector.for_workload(w, W)
    out = binding.make_dqn_outputs(N, L, next_states=False)
    h.run(torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts).cuda(),
          torch.from_numpy(inp.seeds.view(np.int32)).cuda(), N, L, w.gamma, wl.DQN_EPSILON, out)
    assert h.status() == binding.ROLLOUT_OK
    h.close()
    a = out["actions"]
    assert int(a.min()) >= 0 and int(a.max()) < wl.N_ACTIONS
    assert bool((out["td"] >= 0).all()) and bool(torch.isfinite(out["q"]).all())
    # V resets to 1 after every done
    d = out["dones"][:, :-1].bool()
    assert bool((out["states"][:, 1:, 51][d] == 1.0).all())
    idx = np.array([0, 127, 128, 5000, 8191, 12345, 16255, 16383])
    g = {k: v[idx].cpu().numpy() for k, v in out.items()}
    sub = wl.Inputs(inp.features, inp.starts[idx], inp.seeds[idx], inp.weights)
    st = _compare(w, sub, W, {k: v for k, v in g.items()}, np.arange(idx.size), L, wl.DQN_EPSILON)
    assert st["action_replays"] <= 4


def test_full_size_recycling_sampled_episodes():
    """Episode recycling in the benchmark's launch (16384 episodes x 1000 steps):
    eight episodes spread over the CTAs against the oracle with the same option
    (every recycled bar checked through the states' market columns, which are
    compared exactly), and properties of every transition: a fresh portfolio
    after every done, and the episodes do move to new bars."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_reset_heavy_bf16"]
    N, L = w.n_episodes, w.horizon
    inp = wl.generate(w)
    W = wl.dqn_weights(w.seed, 0.05)
    h = binding.DqnCollector.for_workload(w, W)
    h.set_recycle(True)
    out = binding.make_dqn_outputs(N, L, next_states=False)
    h.run(torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts).cuda(),
          torch.from_numpy(inp.seeds.view(np.int32)).cuda(), N, L, w.gamma, wl.DQN_EPSILON, out)
    assert h.status() == binding.ROLLOUT_OK
    h.close()
    a = out["actions"]
    assert int(a.min()) >= 0 and int(a.max()) < wl.N_ACTIONS
    assert bool((out["td"] >= 0).all()) and bool(torch.isfinite(out["q"]).all())
    d = out["dones"][:, :-1].bool()
    assert bool((out["states"][:, 1:, 51][d] == 1.0).all()) and bool((out["states"][:, 1:, 52][d] == 0.0).all())
    idx = np.array([0, 127, 128, 5000, 8191, 12345, 16255, 16383])
    g = {k: v[idx].cpu().numpy() for k, v in out.items()}
    sub = wl.Inputs(inp.features, inp.starts[idx], inp.seeds[idx], inp.weights)
    ref = {}
    st = _compare(w, sub, W, g, np.arange(idx.size), L, wl.DQN_EPSILON, recycle=True, ref_out=ref)
    assert st["action_replays"] <= 4
    plain = inp.starts[idx][:, None].astype(np.int64) + np.arange(L)[None, :]
    assert (ref["bars"] != plain).any()


def test_recycling_at_the_smallest_feature_matrix():
    """Episode recycling with a done on every step (a one-bar time barrier) on the
    smallest feature matrix the horizon allows (n_bars = L + 1, every start 0): each
    draw's range reaches the matrix's end (the last step reads its final row), and
    the collector agrees with the oracle with the same option."""
    import dataclasses
    from rl_experience_collection_gb300 import binding
    w = dataclasses.replace(wl.DQN_WORKLOADS["dqn_tiny_bf16"], max_hold=1)
    N, L = 200, 30
    full = wl.generate(w, n_episodes=N, horizon=L)
    inp = wl.Inputs(np.ascontiguousarray(full.features[:L + 1]), np.zeros(N, np.int32), full.seeds[:N],
                    full.weights)
    W = wl.dqn_weights(17, 0.05)
    status, g = _run(w, inp, W, N, L, 0.3, recycle=True)
    assert status == binding.ROLLOUT_OK
    assert (g["dones"] == 1).all()
    ref = {}
    _compare(w, inp, W, g, np.arange(N), L, 0.3, recycle=True, ref_out=ref)
    bars = ref["bars"]
    assert (bars + (L - np.arange(L))[None, :] <= L).all()      # every next bar inside the matrix
    assert (bars[:, 1:] == np.arange(1, L)[None, :]).any()       # some draws reach the top of the range


def test_episodes_at_the_end_of_the_feature_matrix():
    """Episodes starting at the last valid bar (their last step's next bar, the
    next state behind the TD target, is the feature matrix's last row), mixed with
    episodes at bar 0, against the oracle: the rollout's feature fetches, the state
    rows and the target pass's builders all reach the end of the matrix."""
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    N, L = 300, 40
    inp = wl.generate(w, n_episodes=N, horizon=L)
    nb = inp.features.shape[0]
    starts = np.full(N, nb - L - 1, np.int32)
    starts[::3] = 0
    sub = wl.Inputs(inp.features, starts, inp.seeds[:N], inp.weights)
    W = wl.dqn_weights(23, 0.05)
    status, g = _run(w, sub, W, N, L, 0.2)
    assert status == binding.ROLLOUT_OK
    _compare(w, sub, W, g, np.arange(N), L, 0.2)
