"""Shared helpers for the GPU parity tests: run the CUDA path through the
C ABI, run the oracle on the same seeded inputs, compare.

Tolerances (from the workload specification):
  * integers (actions, dones) and the market part of the states: exact;
    where a uniform lies within ACT_BAND of the CDF boundary that separates
    the two actions (or V'-1 within DONE_BAND of a barrier) the oracle adopts
    the CUDA path's decision and counts a replay;
  * log-probs and values: |g - o| <= rtol * max(|o|, 1), rtol 1e-4 (fp32) or
    2e-2 (bf16 / tf32 tensor-core paths), checked teacher-forced per step;
  * rewards, advantages, returns: abs 1e-3 (fp32) or 5e-2 (bf16 / tf32).
"""
from __future__ import annotations

import dataclasses
import os

import numpy as np

from rl_experience_collection_gb300 import workloads as wl

ACT_BAND = 1e-5
DONE_BAND = 1e-6
RTOL = {"fp32": 1e-4, "tf32": 2e-2, "bf16": 2e-2}
ATOL = {"fp32": 1e-3, "tf32": 5e-2, "bf16": 5e-2}
THREADS = max(1, min(16, os.cpu_count() or 1))


def gpu_run(w: wl.Workload, inputs: wl.Inputs, N: int, L: int):
    import torch
    from rl_experience_collection_gb300 import binding
    out = binding.collect(w, inputs, N=N, L=L)
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in out.items()}


def rel_err(g, o):
    return np.abs(g.astype(np.float64) - o.astype(np.float64)) / np.maximum(np.abs(o.astype(np.float64)), 1.0)


def compare(w: wl.Workload, inputs: wl.Inputs, gpu: dict, idx, L: int, quant: str | None = None):
    """Free-running oracle (with replay) on episodes idx against the GPU outputs.
    Returns (oracle outputs, report dict); raises AssertionError on a violation."""
    from oracle import oracle as orc
    dtype = quant or w.dtype
    ref = orc.rollout(w, inputs, idx, horizon=L, quant=dtype, gpu_actions=gpu["actions"],
                      gpu_dones=gpu["dones"], act_band=ACT_BAND, done_band=DONE_BAND, threads=THREADS)
    st = ref["stats"]
    rep = {"episodes": len(idx), "stats": st}
    assert st["action_mismatches"] == 0, f"actions differ outside the replay band: {st}"
    assert st["done_mismatches"] == 0, f"dones differ outside the replay band: {st}"
    sel = np.asarray(idx)
    g = {k: v[sel] for k, v in gpu.items()}
    np.testing.assert_array_equal(g["actions"], ref["actions"])
    np.testing.assert_array_equal(g["dones"], ref["dones"])
    # states: market features and exposure/spread exact, value within f32 rounding
    np.testing.assert_array_equal(g["states"][..., :51], ref["states"][..., :51])
    np.testing.assert_array_equal(g["states"][..., 52:], ref["states"][..., 52:])
    np.testing.assert_allclose(g["states"][..., 51], ref["states"][..., 51], rtol=2e-6, atol=0)
    rtol, atol = RTOL[dtype], ATOL[dtype]
    for k in ("logp", "values"):
        e = rel_err(g[k], ref[k])
        rep[f"max_rel_{k}"] = float(e.max())
        assert e.max() <= rtol, f"{k}: max rel err {e.max():.3g} > {rtol}"
    for k in ("rewards", "adv", "ret"):
        e = np.abs(g[k].astype(np.float64) - ref[k].astype(np.float64))
        rep[f"max_abs_{k}"] = float(e.max())
        assert e.max() <= atol, f"{k}: max abs err {e.max():.3g} > {atol}"
    return ref, rep


def teacher_forced(w: wl.Workload, inputs: wl.Inputs, gpu: dict, pairs, quant: str):
    """Oracle actor/critic on the GPU's own state rows (n, t) in `pairs`.
    Returns max relative errors of log p[action] and V."""
    from oracle import oracle as orc
    from scipy.special import log_softmax
    cfg = orc.make_cfg(w, quant)
    e_lp, e_v = 0.0, 0.0
    for n, t in pairs:
        x = gpu["states"][n, t].astype(np.float64)
        lp = log_softmax(orc.actor(inputs.weights, cfg, x))[gpu["actions"][n, t]]
        v = orc.critic(inputs.weights, cfg, x)
        e_lp = max(e_lp, abs(gpu["logp"][n, t] - lp) / max(abs(lp), 1.0))
        e_v = max(e_v, abs(gpu["values"][n, t] - v) / max(abs(v), 1.0))
    return e_lp, e_v


def invariants(w: wl.Workload, inputs: wl.Inputs, gpu: dict, L: int, gamma=None, lam=None):
    """Properties that hold at any size, checked over every output element."""
    N = gpu["actions"].shape[0]
    a, d = gpu["actions"], gpu["dones"]
    assert a.min() >= 0 and a.max() < wl.N_ACTIONS
    assert set(np.unique(d)) <= {0, 1}
    for k in ("logp", "values", "rewards", "adv", "ret"):
        assert np.all(np.isfinite(gpu[k])), k
    assert np.all(gpu["logp"] <= 1e-6)
    bars = inputs.starts[:N, None] + np.arange(L)[None, :]
    np.testing.assert_array_equal(gpu["states"][..., :51], inputs.features[bars])
    assert np.all(gpu["states"][..., 53] == np.float32(w.spread))
    # reset after done; exposure follows the previous action otherwise
    e_prev = 0.5 * (a[:, :-1] // 9 - 2)
    want_e = np.where(d[:, :-1] == 1, 0.0, e_prev)
    np.testing.assert_array_equal(gpu["states"][:, 1:, 52], want_e.astype(np.float32))
    assert np.all(gpu["states"][:, 0, 52] == 0) and np.all(gpu["states"][:, 0, 51] == 1)
    assert np.all(gpu["states"][:, 1:, 51][d[:, :-1] == 1] == 1)
    # time barrier: at most K steps between dones
    K = w.max_hold
    since = np.zeros(N, np.int64)
    for t in range(L):
        since += 1
        assert np.all(since <= K)
        since[d[:, t] == 1] = 0
    # GAE recurrence and returns
    g = w.gamma if gamma is None else gamma
    lm = w.lam if lam is None else lam
    A, V, R = gpu["adv"].astype(np.float64), gpu["values"].astype(np.float64), gpu["rewards"].astype(np.float64)
    nd = 1.0 - d
    delta = R[:, :-1] + g * V[:, 1:] * nd[:, :-1] - V[:, :-1]
    resid = A[:, :-1] - delta - g * lm * nd[:, :-1] * A[:, 1:]
    if resid.size:
        assert np.abs(resid).max() < 1e-3, np.abs(resid).max()
    np.testing.assert_array_equal(gpu["ret"], (gpu["adv"] + gpu["values"]).astype(np.float32))
