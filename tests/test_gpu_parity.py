"""GPU parity: the CUDA path (through the C ABI) against the oracle on the
same seeded inputs.  Marked gpu; each test builds nothing itself (the session
fixture builds the library once)."""
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


def _sample(N, k, seed=0):
    if k >= N:
        return np.arange(N)
    rng = np.random.default_rng(seed)
    head = np.arange(min(4, N))
    rest = rng.choice(np.arange(4, N), size=k - len(head), replace=False)
    return np.sort(np.concatenate([head, rest, [N - 1]]))


# ------------------------------------------------------------------ small, several tiles, ragged tails

def _dump(w, N):
    """Episodes whose hidden activations are dumped and replayed (tensor-core paths)."""
    return N if w.dtype != "fp32" else 0


@pytest.mark.parametrize("name", ["tiny_fp32", "scaleout_tf32", "reset_heavy_bf16", "ceiling_bf16"])
@pytest.mark.parametrize("N,L", [(130, 37), (1, 1), (1, 2), (129, 3), (33, 130)])
def test_small_shapes_match_oracle(name, N, L):
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    gpu = parity.gpu_run(w, inp, N, L, dump_episodes=_dump(w, N))
    parity.compare(w, inp, gpu, np.arange(N), L)
    parity.invariants(w, inp, gpu, L)


# reset-heavy shapes at which the bf16 path once differed from the oracle outside
# the stated rules (a value 2.008e-2 from mode Q at 300 x 70, an action drawn
# 1.37e-5 from its CDF boundary at 600 x 70): every episode compared
@pytest.mark.parametrize("N,L", [(300, 70), (600, 70), (1000, 70)])
def test_reset_heavy_all_episodes(N, L):
    w = wl.WORKLOADS["reset_heavy_bf16"]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    gpu = parity.gpu_run(w, inp, N, L, dump_episodes=N)
    _, rep = parity.compare(w, inp, gpu, np.arange(N), L)
    print(N, L, rep)
    parity.invariants(w, inp, gpu, L)


# ------------------------------------------------------------------ full workload sizes

# episodes compared at full size (all of them for the fp32 workloads, the first
# 256 -- with their hidden activations replayed -- for the tensor-core ones)
FULL = [("tiny_fp32", 32), ("default_fp32", 128), ("scaleout_tf32", 256), ("reset_heavy_bf16", 256),
        ("ceiling_bf16", 256)]


@pytest.mark.parametrize("name,k", FULL)
def test_workload_matches_oracle(name, k):
    w = wl.WORKLOADS[name]
    inp = wl.generate(w)
    gpu = parity.gpu_run(w, inp, w.n_episodes, w.horizon, dump_episodes=_dump(w, k))
    idx = np.arange(k)
    _, rep = parity.compare(w, inp, gpu, idx, w.horizon)
    print(name, rep)
    parity.invariants(w, inp, gpu, w.horizon)
    # teacher-forced on episodes outside the compared set: the oracle's networks
    # (mode Q, nothing replayed) on the GPU's own state rows
    rng = np.random.default_rng(1)
    pairs = [(int(n), int(t)) for n, t in zip(rng.integers(0, w.n_episodes, 64), rng.integers(0, w.horizon, 64))]
    e_lp, e_v = parity.teacher_forced(w, inp, gpu, pairs, w.dtype)
    assert e_lp <= parity.RTOL[w.dtype] and e_v <= parity.RTOL[w.dtype], (e_lp, e_v)
    if w.dtype != "fp32":
        # against the unrounded definition (float32 weights, exact arithmetic):
        # log-probs within the bf16 tolerance; values as accurate as the exact
        # bf16 / tf32 network itself (mode Q), whose own distance from the
        # unrounded one exceeds 2e-2 in the tail (operand rounding alone)
        pairs = [(int(n), int(t)) for n, t in zip(rng.integers(0, w.n_episodes, 1024),
                                                  rng.integers(0, w.horizon, 1024))]
        acc = parity.unrounded_accuracy(w, inp, gpu, pairs)
        print(name, "vs unrounded oracle:", acc)
        assert acc["logp_max"] <= parity.RTOL[w.dtype], acc
        assert acc["value_rms"] <= 1.1 * acc["modeq_value_rms"] + 1e-6, acc


# ------------------------------------------------------------------ sampler through the kernel

@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_sampler_chi_squared_through_kernel(dtype):
    from scipy import stats
    w = dataclasses.replace(wl.WORKLOADS["reset_heavy_bf16"], dtype=dtype)
    N, L = 1000, 1000
    inp = wl.generate(w, n_episodes=N, horizon=L)
    views = wl.weight_views(inp.weights, w.critic_h)
    views["actor2.w"][:] = 0.0                         # logits = b3 at every step
    rng = np.random.default_rng(11)
    logits = (rng.standard_normal(wl.N_ACTIONS) * 1.2).astype(np.float32)
    views["actor2.b"][:] = logits
    gpu = parity.gpu_run(w, inp, N, L)
    p = np.exp(logits.astype(np.float64) - logits.max())
    p /= p.sum()
    counts = np.bincount(gpu["actions"].ravel(), minlength=wl.N_ACTIONS)
    chi2, pval = stats.chisquare(counts, p * counts.sum())
    assert pval > 1e-4, (chi2, pval)
    # the draws themselves: exact agreement with the oracle's sampler on a few episodes
    parity.compare(w, inp, gpu, [0, 1, 2, N - 1], L)
    np.testing.assert_allclose(gpu["logp"], (logits - logits.max() - np.log(np.exp(logits - logits.max()).sum()))
                               [gpu["actions"]], rtol=0, atol=2e-6)


# ------------------------------------------------------------------ edge cases and errors

@pytest.mark.parametrize("name", ["reset_heavy_bf16", "scaleout_tf32", "tiny_fp32"])
def test_episodes_at_the_end_of_the_feature_matrix(name):
    """Episodes starting at the last valid bar (their last step's next bar is the
    feature matrix's last row), mixed with episodes at bar 0: the rollout's row
    gathers, the value phase's staged feature runs and the state rows all reach
    the end of the matrix, and every episode matches the oracle."""
    w = wl.WORKLOADS[name]
    N, L = 130, 40
    inp = wl.generate(w, n_episodes=N, horizon=L)
    nb = inp.features.shape[0]
    inp.starts[:] = nb - L - 1
    inp.starts[::3] = 0
    gpu = parity.gpu_run(w, inp, N, L, dump_episodes=_dump(w, N))
    parity.compare(w, inp, gpu, np.arange(N), L)
    parity.invariants(w, inp, gpu, L)


def test_out_of_range_start_sets_status_and_zeroes_episode():
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["tiny_fp32"]
    N, L = 40, 25
    inp = wl.generate(w, n_episodes=N, horizon=L)
    inp.starts[5] = w.n_bars - L            # one past the last valid start
    inp.starts[7] = -3
    h = binding.Rollout.for_workload(w, inp.weights)
    feats = torch.from_numpy(inp.features).cuda()
    out = binding.make_outputs(N, L)
    h.run(feats, torch.from_numpy(inp.starts).cuda(), torch.from_numpy(inp.seeds.view(np.int32)).cuda(), N, L,
          w.gamma, w.lam, out)
    assert h.status() == binding.ROLLOUT_ERR_RANGE
    gpu = {k: v.cpu().numpy() for k, v in out.items()}
    for n in (5, 7):
        for k in binding.OUTPUTS:
            assert not np.any(gpu[k][n]), (n, k)
    ok = [n for n in range(N) if n not in (5, 7)]
    parity.compare(w, inp, gpu, ok, L)
    # the handle stays usable and the next clean run reports OK
    inp2 = wl.generate(w, n_episodes=N, horizon=L)
    h.run(feats, torch.from_numpy(inp2.starts).cuda(), torch.from_numpy(inp2.seeds.view(np.int32)).cuda(), N, L,
          w.gamma, w.lam, out)
    assert h.status() == binding.ROLLOUT_OK
    h.close()


def test_argument_validation():
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["tiny_fp32"]
    N, L = 8, 10
    inp = wl.generate(w, n_episodes=N, horizon=L)
    h = binding.Rollout.for_workload(w, inp.weights)
    feats = torch.from_numpy(inp.features).cuda()
    st = torch.from_numpy(inp.starts).cuda()
    sd = torch.from_numpy(inp.seeds.view(np.int32)).cuda()
    out = binding.make_outputs(N, L)
    ptrs = [feats.data_ptr(), st.data_ptr(), sd.data_ptr()] + [out[k].data_ptr() for k in binding.OUTPUTS]
    assert h.run_raw(ptrs, N, L, 0.99, 0.95) == binding.ROLLOUT_OK
    assert h.status() == binding.ROLLOUT_OK
    bad = list(ptrs)
    bad[3] = 0
    assert h.run_raw(bad, N, L, 0.99, 0.95) == binding.ROLLOUT_ERR_INVALID
    bad = list(ptrs)
    bad[4] += 4                                        # misaligned
    assert h.run_raw(bad, N, L, 0.99, 0.95) == binding.ROLLOUT_ERR_INVALID
    assert h.run_raw(ptrs, N, L, 1.5, 0.95) == binding.ROLLOUT_ERR_INVALID
    assert h.run_raw(ptrs, N, L, 0.99, float("nan")) == binding.ROLLOUT_ERR_INVALID
    assert h.run_raw(ptrs, 0, L, 0.99, 0.95) == binding.ROLLOUT_ERR_INVALID
    assert h.run_raw(ptrs, N, w.n_bars, 0.99, 0.95) == binding.ROLLOUT_ERR_INVALID
    assert "gamma" in binding.last_error() or "L=" in binding.last_error() or binding.last_error()
    h.close()
    d = binding.make_dims(w)
    d.actor_h1 = 100
    with pytest.raises(binding.RolloutError) as ei:
        binding.Rollout(inp.weights, d)
    assert ei.value.code == binding.ROLLOUT_ERR_UNSUPPORTED
    d = binding.make_dims(w)
    bad_w = inp.weights.copy()
    bad_w[3] = np.nan
    with pytest.raises(binding.RolloutError) as ei:
        binding.Rollout(bad_w, d)
    assert ei.value.code == binding.ROLLOUT_ERR_INVALID


def test_set_weights_changes_the_policy():
    w = wl.WORKLOADS["reset_heavy_bf16"]
    N, L = 64, 20
    inp = wl.generate(w, n_episodes=N, horizon=L)
    from rl_experience_collection_gb300 import binding
    h = binding.Rollout.for_workload(w, inp.weights)
    a1 = binding.collect(w, inp, N, L, handle=h)["actions"].cpu().numpy()
    w2 = inp.weights.copy()
    views = wl.weight_views(w2, w.critic_h)
    views["actor2.w"][:] = 0
    views["actor2.b"][:] = -50
    views["actor2.b"][7] = 50
    h.set_weights(w2)
    a2 = binding.collect(w, dataclasses.replace(inp, weights=w2), N, L, handle=h)["actions"].cpu().numpy()
    assert np.all(a2 == 7) and not np.all(a1 == 7)
    h.close()


# ------------------------------------------------------------------ the activation dump itself

@pytest.mark.parametrize("name", ["scaleout_tf32", "reset_heavy_bf16", "ceiling_bf16"])
def test_activation_dump_changes_no_output(name):
    """A run of the dumping test builds gives every output of a normal run bit for
    bit and writes every operand of the dumped episodes (the array is
    NaN-filled before the run), and only the columns each row has."""
    w = wl.WORKLOADS[name]
    N, L, k = 200, 33, 70
    inp = wl.generate(w, n_episodes=N, horizon=L)
    plain = parity.gpu_run(w, inp, N, L)
    dumped = parity.gpu_run(w, inp, N, L, dump_episodes=k)
    for key in plain:
        np.testing.assert_array_equal(dumped[key], plain[key], err_msg=key)
    H = dumped["hidden"]
    IN = 64
    ha, hc, hw = IN, IN + 128 + 64, H.shape[-1]
    assert H.shape == (k, L + 1, hc + sum(w.critic_h) + 64)
    assert np.all(np.isfinite(H[:, :L, :54])) and np.all(np.isfinite(H[:, :L, ha:])), "a step row was left unwritten"
    assert np.all(np.isnan(H[:, :, 54:IN]))
    assert np.all(np.isfinite(H[:, L, :54])) and np.all(np.isfinite(H[:, L, hc:hw - 64])), \
        "a bootstrap row was left unwritten"
    assert np.all(np.isnan(H[:, L, ha:hc])) and np.all(np.isnan(H[:, L, hw - 64:]))
    assert np.all(H[:, :, ha:][np.isfinite(H[:, :, ha:])] >= 0)      # hidden layers: after ReLU
    # the state input is the state row rounded to the operand format
    x = dumped["states"][:k].astype(np.float32).view(np.uint32)
    if w.dtype == "bf16":
        want = ((x + 0x7FFF + ((x >> 16) & 1)) & 0xFFFF0000).view(np.float32)
    else:
        want = ((x + 0x1000) & 0xFFFFE000).view(np.float32)        # tf32, nearest ties away
    np.testing.assert_array_equal(H[:, :L, :54], want)
