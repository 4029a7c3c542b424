"""rollout_run_host: the host-buffer entry point.  Its outputs must equal
rollout_run's bit for bit (the same kernels on the same inputs; rollout_run
itself is compared with the oracle in test_gpu_parity), satisfy the
any-size invariants, and honour NULL outputs, pageable host memory and a
device staging area that grows between calls."""
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


def _host_outputs(N, L, pinned=True, names=None):
    import torch
    from rl_experience_collection_gb300 import binding
    names = binding.OUTPUTS if names is None else names
    dev = binding.make_outputs(N, L, device="cpu")
    return {k: (dev[k].pin_memory() if pinned else dev[k]) for k in names}


def _device_run(h, inp, N, L, w):
    import torch
    from rl_experience_collection_gb300 import binding
    out = binding.make_outputs(N, L)
    h.run(torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts[:N]).cuda(),
          torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda(), N, L, w.gamma, w.lam, out)
    assert h.status() == binding.ROLLOUT_OK
    return {k: v.cpu().numpy() for k, v in out.items()}


@pytest.mark.parametrize("name,N,L", [("reset_heavy_bf16", 300, 70), ("scaleout_tf32", 130, 37),
                                      ("tiny_fp32", 65, 20), ("ceiling_bf16", 129, 33)])
def test_host_entry_equals_device_entry(name, N, L):
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    h = binding.Rollout.for_workload(w, inp.weights, n_bars=inp.features.shape[0])
    ref = _device_run(h, inp, N, L, w)
    feats = torch.from_numpy(inp.features).pin_memory()
    starts = torch.from_numpy(inp.starts[:N]).pin_memory()
    seeds = torch.from_numpy(inp.seeds[:N].view(np.int32)).pin_memory()
    out = _host_outputs(N, L)
    h.run_host(feats, starts, seeds, N, L, w.gamma, w.lam, out)
    torch.cuda.current_stream().synchronize()
    assert h.status() == binding.ROLLOUT_OK
    got = {k: v.numpy() for k, v in out.items()}
    for k in binding.OUTPUTS:
        np.testing.assert_array_equal(got[k], ref[k], err_msg=k)
    parity.invariants(w, inp, got, L)
    h.close()


def test_partial_outputs_pageable_memory_and_growing_staging():
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["reset_heavy_bf16"]
    inp = wl.generate(w, n_episodes=260, horizon=90)
    h = binding.Rollout.for_workload(w, inp.weights, n_bars=inp.features.shape[0])
    # small first, then larger (the staging area grows), then small again
    for N, L in [(40, 9), (260, 90), (129, 33)]:
        ref = _device_run(h, inp, N, L, w)
        names = ("states", "adv", "dones")                       # the others are not copied back
        out = _host_outputs(N, L, pinned=False, names=names)      # pageable: copies complete before return
        h.run_host(np.ascontiguousarray(inp.features), np.ascontiguousarray(inp.starts[:N]),
                   np.ascontiguousarray(inp.seeds[:N]), N, L, w.gamma, w.lam, out)
        torch.cuda.current_stream().synchronize()
        assert h.status() == binding.ROLLOUT_OK
        for k in names:
            np.testing.assert_array_equal(out[k].numpy(), ref[k], err_msg=f"{k} at N={N}, L={L}")
    h.close()


def test_host_entry_validation():
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["reset_heavy_bf16"]
    inp = wl.generate(w, n_episodes=8, horizon=5)
    h = binding.Rollout.for_workload(w, inp.weights, n_bars=inp.features.shape[0])
    out = _host_outputs(8, 5, pinned=False)
    with pytest.raises(binding.RolloutError) as ei:
        h.run_host(inp.features, None, inp.seeds[:8], 8, 5, w.gamma, w.lam, out)
    assert ei.value.code == binding.ROLLOUT_ERR_INVALID
    with pytest.raises(binding.RolloutError) as ei:
        h.run_host(inp.features, inp.starts[:8], inp.seeds[:8], 8, 5, 1.5, w.lam, out)
    assert ei.value.code == binding.ROLLOUT_ERR_INVALID
    h.close()
