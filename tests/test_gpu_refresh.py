"""rollout_set_weights_device: refreshing a handle from device weights must
leave it converted exactly as rollout_set_weights (host) does, for every
precision and both critic widths, so the two handles' collections are equal
bit for bit (the host path itself is compared with the oracle in
test_gpu_parity).  Also the closed loop collect -> PPO update -> refresh with
no host copy of the weights."""
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


def _run(h, inp, N, L, w):
    import torch
    from rl_experience_collection_gb300 import binding
    out = binding.make_outputs(N, L)
    h.run(torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts[:N]).cuda(),
          torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda(), N, L, w.gamma, w.lam, out)
    assert h.status() == binding.ROLLOUT_OK
    return {k: v.cpu().numpy() for k, v in out.items()}


def _new_weights(w0, seed):
    """Every weight changed: a fresh draw at the same scale, with one weight in 64
    set on a bf16 rounding tie (low 16 bits 0x8000) and one in 64 on a tf32 tie
    (low 13 bits 0x1000), where the two rounding rules part."""
    rng = np.random.default_rng(seed)
    w1 = (w0 + 0.05 * rng.standard_normal(w0.size)).astype(np.float32)
    u = w1.view(np.uint32)
    u[0::64] = (u[0::64] & 0xFFFF0000) | 0x8000
    u[1::64] = (u[1::64] & 0xFFFFE000) | 0x1000
    return w1


@pytest.mark.parametrize("name,N,L", [("tiny_fp32", 40, 25), ("scaleout_tf32", 130, 30),
                                      ("reset_heavy_bf16", 300, 40), ("ceiling_bf16", 129, 24)])
def test_device_refresh_equals_host_refresh(name, N, L):
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    inp = wl.generate(w, n_episodes=N, horizon=L)
    w1 = _new_weights(inp.weights, 5)
    nb = inp.features.shape[0]
    host = binding.Rollout.for_workload(w, inp.weights, n_bars=nb)
    dev = binding.Rollout.for_workload(w, inp.weights, n_bars=nb)
    before = _run(dev, inp, N, L, w)
    host.set_weights(w1)
    dev.set_weights_device(torch.from_numpy(w1).cuda())
    a, b = _run(host, inp, N, L, w), _run(dev, inp, N, L, w)
    fresh = binding.Rollout.for_workload(w, w1, n_bars=nb)
    c = _run(fresh, inp, N, L, w)
    for k in binding.OUTPUTS:
        np.testing.assert_array_equal(a[k], b[k], err_msg=k)
        np.testing.assert_array_equal(a[k], c[k], err_msg=k)
    assert not np.array_equal(before["values"], b["values"])     # the refresh took effect
    # and back: the original weights give the original collection
    dev.set_weights_device(torch.from_numpy(inp.weights).cuda())
    again = _run(dev, inp, N, L, w)
    for k in binding.OUTPUTS:
        np.testing.assert_array_equal(before[k], again[k], err_msg=k)
    for h in (host, dev, fresh):
        h.close()


@pytest.mark.parametrize("name", ["tiny_fp32", "reset_heavy_bf16"])
def test_collect_update_refresh_loop_without_host_weights(name):
    """Two rounds of collect -> 3 PPO steps -> refresh from the trainer's own device
    weights, against the same loop refreshed from a host copy of the weights."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    N, L = 64, 24
    inp = wl.generate(w, n_episodes=N, horizon=L)
    nb = inp.features.shape[0]
    feats = torch.from_numpy(inp.features).cuda()
    starts = torch.from_numpy(inp.starts[:N]).cuda()
    seeds = torch.from_numpy(inp.seeds[:N].view(np.int32)).cuda()
    idx = torch.from_numpy(np.random.default_rng(3).permutation(N * L)[:3 * 128].astype(np.int32)).cuda()

    def loop(device_refresh):
        h = binding.Rollout.for_workload(w, inp.weights, n_bars=nb)
        tr = binding.PpoTrainer.for_workload(w, inp.weights)
        outs = []
        for _ in range(2):
            out = binding.make_outputs(N, L)
            h.run(feats, starts, seeds, N, L, w.gamma, w.lam, out)
            tr.update(out["states"].reshape(-1, wl.STATE_DIM), out["actions"].reshape(-1), out["logp"].reshape(-1),
                      out["adv"].reshape(-1), out["ret"].reshape(-1), idx, 3, 128)
            if device_refresh:
                h.set_weights_device(tr.device_weights())
            else:
                h.set_weights(tr.weights())
            outs.append({k: v.cpu().numpy() for k, v in out.items()})
        out = binding.make_outputs(N, L)
        h.run(feats, starts, seeds, N, L, w.gamma, w.lam, out)
        outs.append({k: v.cpu().numpy() for k, v in out.items()})
        assert h.status() == binding.ROLLOUT_OK and tr.status() == binding.ROLLOUT_OK
        final = tr.weights()
        h.close()
        tr.close()
        return outs, final

    a, wa = loop(True)
    b, wb = loop(False)
    np.testing.assert_array_equal(wa, wb)
    assert not np.array_equal(wa, inp.weights)
    for r in range(3):
        for k in binding.OUTPUTS:
            np.testing.assert_array_equal(a[r][k], b[r][k], err_msg=f"{r} {k}")


def test_device_refresh_rejects_bad_arguments():
    import ctypes as C
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS["tiny_fp32"]
    inp = wl.generate(w, n_episodes=4, horizon=4)
    h = binding.Rollout.for_workload(w, inp.weights, n_bars=inp.features.shape[0])
    L = binding.lib()
    assert L.rollout_set_weights_device(h._h, None, None) == binding.ROLLOUT_ERR_INVALID
    t = torch.from_numpy(inp.weights).cuda()
    assert L.rollout_set_weights_device(h._h, C.c_void_p(t.data_ptr() + 2), None) == binding.ROLLOUT_ERR_INVALID
    with pytest.raises(ValueError):
        h.set_weights_device(torch.from_numpy(inp.weights))          # a host tensor
    with pytest.raises(ValueError):
        h.set_weights_device(t.double())
    h.close()
