"""The DQN flow of the pages on the device, end to end: a collection by the DQN
collector (include/dqn.h) goes into the prioritised replay buffer (include/per.h)
with its TD errors as priorities, and a training batch is drawn, with no host
round trip between the calls.  Each component is compared with its oracle in
its own test file; this checks that they compose: the rows the buffer gives
back are the collector's, and the priorities are the update rule applied to the
collector's TD errors."""
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


def test_collect_insert_prioritise_sample():
    import torch
    from rl_experience_collection_gb300 import binding
    from oracle import per
    w = wl.DQN_WORKLOADS["dqn_tiny_bf16"]
    N, L = 256, 50
    T = N * L
    inp = wl.generate(w, n_episodes=N, horizon=L)
    col = binding.DqnCollector.for_workload(w, wl.dqn_weights(2, 0.05), n_bars=inp.features.shape[0])
    out = binding.make_dqn_outputs(N, L)
    col.run(torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts).cuda(),
            torch.from_numpy(inp.seeds.view(np.int32)).cuda(), N, L, w.gamma, 0.1, out)
    buf = binding.PerBuffer(T + 1000, wl.STATE_DIM)
    flat = lambda k, *shape: out[k].reshape(*shape)
    buf.insert(flat("states", T, wl.STATE_DIM), flat("next_states", T, wl.STATE_DIM), flat("actions", T),
               flat("rewards", T), flat("dones", T).to(torch.uint8))
    slots = torch.arange(T, dtype=torch.int32, device="cuda")
    buf.update(slots, flat("td", T), alpha=0.6, eps=1e-6)
    batch = buf.make_batch(512)
    buf.sample(512, 0.4, 5, 0, batch)
    assert col.status() == binding.ROLLOUT_OK and buf.status() == binding.ROLLOUT_OK
    col.close()
    g = {k: v.cpu().numpy() for k, v in out.items()}
    # the priorities are the update rule on the collector's TD errors
    ref = per.Replay(T + 1000, 0)
    ref.insert(None, None, g["actions"].reshape(-1), g["rewards"].reshape(-1),
               g["dones"].reshape(-1).astype(np.uint8))
    ref.update(np.arange(T), g["td"].reshape(-1), 0.6, 1e-6)
    pr, m = buf.priorities()
    diff = pr[:T].view(np.int32).astype(np.int64) - ref.prio[:T].view(np.int32).astype(np.int64)
    assert np.abs(diff).max() <= 1 and m == ref.max_prio
    # the batch holds the collector's transitions at the drawn slots
    b = {k: v.cpu().numpy() for k, v in batch.items()}
    idx = b["indices"].astype(np.int64)
    assert ((idx >= 0) & (idx < T)).all()
    np.testing.assert_array_equal(b["states"], g["states"].reshape(T, -1)[idx])
    np.testing.assert_array_equal(b["next_states"], g["next_states"].reshape(T, -1)[idx])
    np.testing.assert_array_equal(b["actions"], g["actions"].reshape(-1)[idx])
    np.testing.assert_array_equal(b["rewards"], g["rewards"].reshape(-1)[idx])
    np.testing.assert_array_equal(b["dones"], g["dones"].reshape(-1)[idx].astype(np.uint8))
    # and the draw is the oracle's on these priorities
    oi, ow, _, _ = ref.sample(512, 0.4, 5, 0, replay=b["indices"], band=1e-12)
    np.testing.assert_array_equal(b["indices"], oi)
    np.testing.assert_allclose(b["weights"], ow, rtol=1e-5)
    buf.close()
