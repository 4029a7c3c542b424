"""Failure detection without a GPU fault: an injected device-allocation failure
in rollout_create (and in rollout_run_host's staging) must return
ROLLOUT_ERR_NOMEM and leave nothing allocated; NaN weights installed through
rollout_set_weights_device (which does not check finiteness) must give NaN
outputs and a clean status, with no hang, and the handle must recover when
finite weights come back."""
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


@pytest.mark.parametrize("name", ["tiny_fp32", "scaleout_tf32", "reset_heavy_bf16", "ceiling_bf16"])
def test_failed_allocation_in_create_returns_nomem_and_leaks_nothing(name):
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=8, horizon=8)
    torch.cuda.synchronize()
    base = binding.test_alloc(0)
    free0 = torch.cuda.mem_get_info()[0]
    failures = 0
    try:
        for k in range(1, 64):
            binding.test_alloc(k)
            try:
                h = binding.Rollout.for_workload(w, inp.weights)
            except binding.RolloutError as e:
                assert e.code == binding.ROLLOUT_ERR_NOMEM, (k, e)
                assert binding.test_alloc(0) == base, f"allocation {k} failed and the create leaked"
                failures += 1
                continue
            # k is past the last allocation: the create succeeded
            assert binding.test_alloc(0) > base
            h.close()
            break
        else:
            pytest.fail("rollout_create kept failing")
    finally:
        binding.test_alloc(0)
    assert failures >= 3, failures              # status word, div table, weights at least
    assert binding.test_alloc(0) == base
    torch.cuda.synchronize()
    assert abs(torch.cuda.mem_get_info()[0] - free0) <= 4 << 20


def test_failed_staging_allocation_in_run_host_leaves_the_handle_usable():
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["reset_heavy_bf16"]
    N, L = 64, 12
    inp = wl.generate(w, n_episodes=N, horizon=L)
    h = binding.Rollout.for_workload(w, inp.weights)
    hf, hs = torch.from_numpy(inp.features), torch.from_numpy(inp.starts)
    hd = torch.from_numpy(inp.seeds.view(np.int32))
    hout = {k: torch.empty(v.shape, dtype=v.dtype) for k, v in binding.make_outputs(N, L, "cpu").items()}
    live = binding.test_alloc(1)
    try:
        with pytest.raises(binding.RolloutError) as ei:
            h.run_host(hf, hs, hd, N, L, w.gamma, w.lam, hout)
        assert ei.value.code == binding.ROLLOUT_ERR_NOMEM
        assert binding.test_alloc(0) == live
    finally:
        binding.test_alloc(0)
    h.run_host(hf, hs, hd, N, L, w.gamma, w.lam, hout)
    torch.cuda.synchronize()
    assert h.status() == binding.ROLLOUT_OK
    ref = binding.collect(w, inp, N, L)
    for k in binding.OUTPUTS:
        np.testing.assert_array_equal(hout[k].numpy(), ref[k].cpu().numpy(), err_msg=k)
    h.close()


@pytest.mark.parametrize("name", ["scaleout_tf32", "reset_heavy_bf16"])
def test_nan_weights_propagate_without_a_hang(name):
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    N, L = 300, 40
    inp = wl.generate(w, n_episodes=N, horizon=L)
    h = binding.Rollout.for_workload(w, inp.weights)
    base = {k: v.cpu().numpy() for k, v in binding.collect(w, inp, N, L, handle=h).items()}

    def run_with(weights):
        dw = torch.from_numpy(np.ascontiguousarray(weights, np.float32)).cuda()
        h.set_weights_device(dw)
        t0 = time.perf_counter()
        out = binding.collect(w, inp, N, L, handle=h)        # raises on a non-OK device status
        torch.cuda.synchronize()
        assert time.perf_counter() - t0 < 60
        assert h.status() == binding.ROLLOUT_OK
        return {k: v.cpu().numpy() for k, v in out.items()}

    # a NaN critic weight: every value is NaN (so are advantages and returns); the
    # actor, the sampler and the environment are untouched
    bad = inp.weights.copy()
    wl.weight_views(bad, w.critic_h)["critic0.w"][0, 0] = np.nan
    got = run_with(bad)
    assert np.all(np.isnan(got["values"])) and np.all(np.isnan(got["adv"])) and np.all(np.isnan(got["ret"]))
    for k in ("states", "actions", "logp", "dones", "rewards"):
        np.testing.assert_array_equal(got[k], base[k], err_msg=k)

    # a NaN actor weight: the logits are NaN, no running sum ever exceeds u * S,
    # so every draw takes the last action and every log-probability is NaN
    bad = inp.weights.copy()
    wl.weight_views(bad, w.critic_h)["actor2.w"][0, 0] = np.nan
    got = run_with(bad)
    assert np.all(got["actions"] == wl.N_ACTIONS - 1) and np.all(np.isnan(got["logp"]))

    # finite weights again: the next run equals the first bit for bit
    got = run_with(inp.weights)
    for k in binding.OUTPUTS:
        np.testing.assert_array_equal(got[k], base[k], err_msg=k)
    h.close()
