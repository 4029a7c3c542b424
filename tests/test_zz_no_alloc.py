"""rollout_run_static: the entry point for callers that cannot allocate device
memory (for example code running under CUDA graph capture, or a host that
fixes the library's device-memory budget at start-up).  It must give the same
results as rollout_run, call after call, while taking the value phase's
activation scratch from the library's fixed device array.

This file is collected last on purpose: it runs after every other test, and
also passes on its own in a fresh process."""
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


@pytest.mark.parametrize("name,N,L", [("scaleout_tf32", 300, 64), ("ceiling_bf16", 200, 40)])
def test_static_scratch_entry_matches_rollout_run(name, N, L):
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    h = binding.Rollout.for_workload(w, inp.weights)
    feats = torch.from_numpy(inp.features).cuda()
    starts = torch.from_numpy(inp.starts).cuda()
    seeds = torch.from_numpy(inp.seeds.view(np.int32)).cuda()
    ref = binding.make_outputs(N, L)
    h.run(feats, starts, seeds, N, L, w.gamma, w.lam, ref)
    assert h.status() == binding.ROLLOUT_OK
    ref = {k: v.cpu().numpy() for k, v in ref.items()}
    for call in range(2):                       # twice in a row: the shared array keeps old contents
        out = binding.make_outputs(N, L)
        for v in out.values():
            v.fill_(7)
        h.run_static(feats, starts, seeds, N, L, w.gamma, w.lam, out)
        assert h.status() == binding.ROLLOUT_OK, binding.last_error()
        got = {k: v.cpu().numpy() for k, v in out.items()}
        # every tile's arithmetic is independent of the CTA and grid that run it,
        # so the two entry points agree bit for bit; a tolerance could hide two
        # CTAs overlapping in the shared array
        for k in binding.OUTPUTS:
            np.testing.assert_array_equal(got[k], ref[k], err_msg=f"call {call}: {k}")
    h.close()
