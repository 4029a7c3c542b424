"""The on-device PPO update (include/ppo.h) against the oracle (oracle/ppo.c)
on the same tuples (collected by the GPU path) and the same seeded
mini-batch indices."""
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
    from oracle import ppo
    ppo.build()


@pytest.fixture(scope="module")
def tuples():
    """A small fp32 collection: 40 episodes x 30 steps."""
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.generate(w, n_episodes=40, horizon=30)
    g = parity.gpu_run(w, inp, 40, 30)
    return w, inp, g


def _device(g):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(g[k].reshape(-1, 54) if k == "states" else g[k].reshape(-1))).cuda()
            for k in ("states", "actions", "logp", "adv", "ret")]


N_TRAINED = 383150   # actor 18,221 + critic 364,929 (the standard critic)


def _layer_bounds(critic_h):
    sizes = [54 * 128, 128, 128 * 64, 64, 64 * 45, 45]
    prev = 54
    for o in list(critic_h) + [1]:
        sizes += [prev * o, o]
        prev = o
    return np.cumsum([0] + sizes)


def _teacher_forced(w, inp, g, idx, n_steps, B, hp_kw):
    """Runs the GPU trainer one step at a time and checks each step in two parts.
    (1) The gradient: ppo_gradient at the GPU's current weights against the oracle's
    loss_grad at the same weights, layer by layer (relative L2 error), and the loss
    statistics.  (2) The optimizer: the oracle's clip + Adam fed the GPU's own gradient
    (its moments follow the same gradients) against the GPU's step, element by element.
    Comparing free-running trajectories instead would amplify float32-level gradient
    differences: Adam normalises each element.  Each step takes the next B rows of the
    seeded order idx, unfiltered; where a hidden pre-activation lies within the float32
    products' error of the ReLU kink, the oracle adopts the side the GPU took (a replay,
    like an action drawn within rounding of a CDF boundary) and any other difference
    fails the step."""
    import torch
    from rl_experience_collection_gb300 import binding
    from oracle import ppo
    hp_o = ppo.Hyper(**hp_kw)
    hp_g = binding.PpoHparams.make(**hp_kw)
    shape = ppo.shape_of(w.critic_h)
    bounds = _layer_bounds(w.critic_h)
    b = ppo.Batch(g["states"], g["actions"], g["logp"], g["adv"], g["ret"])
    states, actions, logp, adv, ret = _device(g)
    tr = binding.PpoTrainer.for_workload(w, inp.weights)
    m = np.zeros(N_TRAINED)
    v = np.zeros(N_TRAINED)
    w_prev = inp.weights.astype(np.float32)
    grad_dev = torch.zeros(N_TRAINED, dtype=torch.float32, device="cuda")
    replays = 0
    for k in range(n_steps):
        rows = np.ascontiguousarray(idx[k * B:(k + 1) * B])
        assert len(rows) == B
        rows_dev = torch.from_numpy(rows).cuda()
        st_g = torch.zeros(4, dtype=torch.float32, device="cuda")
        tr.gradient(states, actions, logp, adv, ret, rows_dev, B, grad_dev, st_g, hp_g)
        act = tr.activations(B)
        st_dev = torch.zeros((1, 5), dtype=torch.float32, device="cuda")
        tr.update(states, actions, logp, adv, ret, rows_dev, 1, B, hp_g, st_dev)
        w_gpu = tr.weights()
        g_gpu = grad_dev.cpu().numpy().astype(np.float64)
        st_gpu = st_dev.cpu().numpy()[0]
        np.testing.assert_array_equal(st_g.cpu().numpy(), st_gpu[:4])
        # (1) gradient and statistics at the same weights, the GPU's ReLU sides replayed
        p = w_prev[:N_TRAINED].astype(np.float64)
        st_o, g_o, rep, mis = ppo.loss_grad_replay(p, shape, hp_o, b, rows, act)
        assert mis == 0, (k, mis, "ReLU sides differ beyond the products' float32 error")
        replays += rep
        for lo, hi in zip(bounds[:-1], bounds[1:]):
            ref = np.linalg.norm(g_o[lo:hi])
            assert np.linalg.norm(g_gpu[lo:hi] - g_o[lo:hi]) <= 1e-3 * ref + 1e-9, (k, lo, hi)
            assert np.max(np.abs(g_gpu[lo:hi] - g_o[lo:hi])) <= 1e-3 * ref + 1e-9, (k, lo, hi)
        assert np.linalg.norm(g_gpu - g_o) <= 2e-4 * np.linalg.norm(g_o), k
        for j in (0, 1, 3):
            assert abs(st_gpu[j] - st_o[j]) <= 2e-4 * abs(st_o[j]) + 1e-6, (k, j, st_gpu[j], st_o[j])
        assert abs(st_gpu[2] - st_o[2]) <= 1.0 / B + 1e-7
        # (2) clip + Adam on the GPU's gradient
        p0 = p.copy()
        norm = ppo.adam_step(p, g_gpu.copy(), m, v, k + 1, hp_o)
        assert abs(st_gpu[4] - norm) <= 1e-5 * norm, (k, st_gpu[4], norm)
        d_gpu = w_gpu[:N_TRAINED].astype(np.float64) - p0
        d_o = p - p0
        tol = 1e-4 * hp_o.lr + 1e-5 * hp_o.weight_decay * np.abs(p0) + 1e-9
        bad = np.abs(d_gpu - d_o) > tol
        assert not bad.any(), (k, np.flatnonzero(bad)[:10], d_gpu[bad][:5], d_o[bad][:5])
        np.testing.assert_array_equal(w_gpu[N_TRAINED:], inp.weights[N_TRAINED:])   # curiosity untouched
        w_prev = w_gpu
    assert tr.status() == binding.ROLLOUT_OK
    tr.close()
    print("ReLU replays", replays)


def test_update_matches_oracle_small_batches(tuples):
    w, inp, g = tuples
    T = g["actions"].size
    idx = np.random.default_rng(11).permutation(T).astype(np.int32)
    _teacher_forced(w, inp, g, idx, 3, 64, dict(lr=3e-4, max_grad_norm=0.5))


def test_update_matches_oracle_batch_512_without_clip_with_decay(tuples):
    w, inp, g = tuples
    T = g["actions"].size
    idx = np.random.default_rng(12).permutation(T).astype(np.int32)
    _teacher_forced(w, inp, g, idx, 2, 512,
                    dict(lr=1e-3, max_grad_norm=0.0, weight_decay=1e-4, clip_eps=0.1, value_coef=0.5))


@pytest.mark.parametrize("n", [3, 6])
def test_multi_step_call_equals_single_steps(tuples, n):
    """n steps in one call (3: launched directly; 6: one captured step replayed)
    equal n calls of one step; after reset_optimizer a trainer repeats its first step."""
    import torch
    from rl_experience_collection_gb300 import binding
    w, inp, g = tuples
    T = g["actions"].size
    idx = np.random.default_rng(14).permutation(T)[:n * 50].astype(np.int32)
    states, actions, logp, adv, ret = _device(g)
    a = binding.PpoTrainer.for_workload(w, inp.weights)
    st_a = torch.zeros((n, 5), dtype=torch.float32, device="cuda")
    a.update(states, actions, logp, adv, ret, torch.from_numpy(idx).cuda(), n, 50, stats=st_a)
    b = binding.PpoTrainer.for_workload(w, inp.weights)
    st_b = torch.zeros((n, 5), dtype=torch.float32, device="cuda")
    for k in range(n):
        b.update(states, actions, logp, adv, ret, torch.from_numpy(idx[50 * k:50 * k + 50].copy()).cuda(), 1, 50,
                 stats=st_b[k:k + 1])
    np.testing.assert_array_equal(a.weights(), b.weights())
    np.testing.assert_array_equal(st_a.cpu().numpy(), st_b.cpu().numpy())
    # a fresh trainer's first step equals a reset trainer's first step from the same weights
    c = binding.PpoTrainer(a.weights(), binding.make_dims(w))
    a.reset_optimizer()
    first = torch.from_numpy(idx[:50].copy()).cuda()
    a.update(states, actions, logp, adv, ret, first, 1, 50)
    c.update(states, actions, logp, adv, ret, first, 1, 50)
    np.testing.assert_array_equal(a.weights(), c.weights())
    for tr in (a, b, c):
        tr.close()


def test_update_is_deterministic_and_reports_out_of_range_indices(tuples):
    import torch
    from rl_experience_collection_gb300 import binding
    w, inp, g = tuples
    T = g["actions"].size
    idx = np.random.default_rng(13).permutation(T)[:4 * 100].astype(np.int32)
    states, actions, logp, adv, ret = _device(g)
    out = []
    for _ in range(2):
        tr = binding.PpoTrainer.for_workload(w, inp.weights)
        tr.update(states, actions, logp, adv, ret, torch.from_numpy(idx).cuda(), 4, 100)
        assert tr.status() == binding.ROLLOUT_OK
        out.append(tr.weights())
        tr.close()
    np.testing.assert_array_equal(out[0], out[1])
    bad = idx.copy()
    bad[5], bad[150] = -1, T + 7
    tr = binding.PpoTrainer.for_workload(w, inp.weights)
    tr.update(states, actions, logp, adv, ret, torch.from_numpy(bad).cuda(), 2, 100)
    assert tr.status() == binding.ROLLOUT_ERR_RANGE
    assert tr.status() == binding.ROLLOUT_OK            # the status word is read once
    with pytest.raises(binding.RolloutError):
        tr.update(states, actions, logp, adv, ret, torch.from_numpy(idx).cuda(), 1, 5000)   # batch > 4096
    with pytest.raises(binding.RolloutError):
        tr.update(states, actions, logp, adv, ret, torch.from_numpy(idx).cuda(), 1, 10,
                  binding.PpoHparams.make(beta2=1.0))
    tr.close()
