"""The device-side timeout path (include/rollout.h rollout_test_stall,
include/dqn.h dqn_test_stall).

A test build of a kernel leaves CTA 0's first weight stage unfilled, so that
CTA's MMA issuer waits on a barrier that nothing completes.  The bounded wait
must expire (about two seconds), every warp of the CTA must leave and release
its tensor memory, the run must report ROLLOUT_ERR_TIMEOUT, and the handle's
next run must be bit-identical to a run before the stall.  Nothing faults,
traps or hangs: the wait that runs out is the kernel's own bounded wait, and
only the status word carries the failure to the host.

Covered: both value kernels of the PPO collector (the shared-memory-resident
bf16 kernel with the standard critic; the scratch-staged one for tf32 and for
bf16 with the wide critic) and the DQN collector's target pass."""
import time

import numpy as np
import pytest

from rl_experience_collection_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rl_experience_collection_gb300 import build
    build.build()


def _run(h, dev, N, L, w):
    from rl_experience_collection_gb300 import binding
    out = binding.make_outputs(N, L)
    t0 = time.perf_counter()
    h.run(*dev, N, L, w.gamma, w.lam, out)
    status = h.status()                       # synchronises
    return status, time.perf_counter() - t0, {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("name,N,L", [("reset_heavy_bf16", 300, 20), ("scaleout_tf32", 130, 16),
                                      ("ceiling_bf16", 129, 12)])
def test_stalled_value_kernel_times_out_and_handle_recovers(name, N, L):
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    dev = (torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts[:N]).cuda(),
           torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda())
    h = binding.Rollout.for_workload(w, inp.weights, n_bars=inp.features.shape[0])
    s0, _, before = _run(h, dev, N, L, w)
    assert s0 == binding.ROLLOUT_OK

    h.test_stall(True)
    s1, dt, stalled = _run(h, dev, N, L, w)
    assert s1 == binding.ROLLOUT_ERR_TIMEOUT, binding.last_error()
    assert 1.5 < dt < 60.0, dt                 # the wait ran to its limit, then the kernel left
    assert h.status() == binding.ROLLOUT_ERR_TIMEOUT   # the last run's status until the next run
    # the rollout kernel ran before the stalled one: its outputs are untouched
    for k in ("actions", "logp", "dones", "states"):
        np.testing.assert_array_equal(stalled[k], before[k], err_msg=k)
    if name == "reset_heavy_bf16":
        # one CTA per tile here (fewer tiles than SMs): only tile 0's rows
        # (the first 128 of the N x L transitions) lack their values
        tiles = (N * L + N + 127) // 128
        assert tiles < torch.cuda.get_device_properties(0).multi_processor_count
        np.testing.assert_array_equal(stalled["values"].reshape(-1)[128:], before["values"].reshape(-1)[128:])

    h.test_stall(False)
    s2, _, after = _run(h, dev, N, L, w)
    assert s2 == binding.ROLLOUT_OK
    for k in before:
        np.testing.assert_array_equal(after[k], before[k], err_msg=k)
    h.close()


def test_stall_hook_rejects_the_fp32_path():
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.generate(w, n_episodes=4, horizon=4)
    h = binding.Rollout.for_workload(w, inp.weights, n_bars=inp.features.shape[0])
    with pytest.raises(binding.RolloutError):
        h.test_stall(True)
    h.close()


@pytest.mark.parametrize("recycle", [False, True])
def test_stalled_dqn_target_pass_times_out_and_collector_recovers(recycle):
    """The DQN collector's target pass with CTA 0's first weight stage never
    filled: ROLLOUT_ERR_TIMEOUT after the bounded wait (read once: dqn_status
    clears the word), the rollout's outputs complete, the other CTAs' rewards
    and TD errors untouched, and the next run bit-identical; also with episode
    recycling (the target pass's recycling builds)."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    N, L = 130, 12
    inp = wl.generate(w, n_episodes=N, horizon=L)
    dev = (torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts[:N]).cuda(),
           torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda())
    h = binding.DqnCollector.for_workload(w, wl.dqn_weights(3, 0.05), n_bars=inp.features.shape[0])
    h.set_recycle(recycle)

    def run():
        out = binding.make_dqn_outputs(N, L)
        t0 = time.perf_counter()
        h.run(*dev, N, L, w.gamma, 0.1, out)
        st = h.status()
        return st, time.perf_counter() - t0, {k: v.cpu().numpy() for k, v in out.items()}

    s0, _, before = run()
    assert s0 == binding.ROLLOUT_OK
    h.test_stall(True)
    s1, dt, stalled = run()
    assert s1 == binding.ROLLOUT_ERR_TIMEOUT and 1.5 < dt < 60.0, (s1, dt)
    assert h.status() == binding.ROLLOUT_OK                 # cleared by the read
    for k in ("states", "actions", "dones", "q"):
        np.testing.assert_array_equal(stalled[k], before[k], err_msg=k)
    tiles = (N * L + 127) // 128                             # one CTA per tile: CTA 0 has rows 0..127
    assert tiles < torch.cuda.get_device_properties(0).multi_processor_count
    for k in ("rewards", "td"):
        np.testing.assert_array_equal(stalled[k].reshape(-1)[128:], before[k].reshape(-1)[128:], err_msg=k)
    np.testing.assert_array_equal(stalled["next_states"].reshape(N * L, -1)[128:],
                                  before["next_states"].reshape(N * L, -1)[128:])
    h.test_stall(False)
    s2, _, after = run()
    assert s2 == binding.ROLLOUT_OK
    for k in before:
        np.testing.assert_array_equal(after[k], before[k], err_msg=k)
    h.close()
