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

On the tensor-core paths the comparison is against mode Q (operands rounded
like the path's) and, where the path's rounded hidden activations were dumped
(rollout_test_activations), with its rounding decisions replayed: a hidden
value may differ from the oracle's only where the exact pre-activation lies
within the float32 accumulation bound of a rounding boundary; any other
difference is a hidden mismatch and fails the comparison.
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
# With every rounding decision of the path replayed, what is left between the
# two is float32 accumulation (log-softmax, the critic head, the curiosity
# error, GAE): a regression net far inside the tolerances above
REPLAYED_RTOL, REPLAYED_ATOL = 2e-5, 2e-5
THREADS = max(1, min(16, os.cpu_count() or 1))


def gpu_run(w: wl.Workload, inputs: wl.Inputs, N: int, L: int, dump_episodes: int = 0):
    """The CUDA path's outputs as numpy arrays; dump_episodes > 0 (tf32 / bf16)
    adds "hidden", the rounded hidden activations of the first episodes."""
    import torch
    from rl_experience_collection_gb300 import binding
    out = binding.collect(w, inputs, N=N, L=L, dump_episodes=dump_episodes if w.dtype != "fp32" else 0)
    torch.cuda.synchronize()
    res = {k: v.cpu().numpy() for k, v in out.items()}
    del out
    torch.cuda.empty_cache()
    return res


def rel_err(g, o):
    return np.abs(g.astype(np.float64) - o.astype(np.float64)) / np.maximum(np.abs(o.astype(np.float64)), 1.0)


def compare(w: wl.Workload, inputs: wl.Inputs, gpu: dict, idx, L: int, quant: str | None = None):
    """Free-running oracle (with replay) on episodes idx against the GPU outputs.
    Returns (oracle outputs, report dict); raises AssertionError on a violation."""
    from oracle import oracle as orc
    dtype = quant or w.dtype
    hidden = gpu.get("hidden") if dtype == w.dtype else None
    ref = orc.rollout(w, inputs, idx, horizon=L, quant=dtype, gpu_actions=gpu["actions"],
                      gpu_dones=gpu["dones"], act_band=ACT_BAND, done_band=DONE_BAND, threads=THREADS,
                      gpu_hidden=hidden)
    st = ref["stats"]
    rep = {"episodes": len(idx), "stats": st,
           "replayed_hidden": hidden is not None and int(np.max(idx)) < hidden.shape[0]}
    assert st["action_mismatches"] == 0, f"actions differ outside the replay band: {st}"
    assert st["done_mismatches"] == 0, f"dones differ outside the replay band: {st}"
    assert st["hidden_mismatches"] == 0, f"hidden activations differ beyond float32 accumulation error: {st}"
    sel = np.asarray(idx)
    g = {k: v[sel] for k, v in gpu.items()}
    np.testing.assert_array_equal(g["actions"], ref["actions"])
    np.testing.assert_array_equal(g["dones"], ref["dones"])
    # states: market features and exposure/spread exact, value within f32 rounding
    np.testing.assert_array_equal(g["states"][..., :51], ref["states"][..., :51])
    np.testing.assert_array_equal(g["states"][..., 52:], ref["states"][..., 52:])
    np.testing.assert_allclose(g["states"][..., 51], ref["states"][..., 51], rtol=2e-6, atol=0)
    rtol, atol = RTOL[dtype], ATOL[dtype]
    if rep["replayed_hidden"]:
        rtol, atol = REPLAYED_RTOL, REPLAYED_ATOL
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


def unrounded_accuracy(w: wl.Workload, inputs: wl.Inputs, gpu: dict, pairs):
    """Errors |g - u| / max(|u|, 1) of the GPU's log-probs and values against
    the unrounded oracle (float32 weights, exact arithmetic) on the GPU's own
    state rows, next to those of mode Q (the exact reduced-precision network)."""
    from oracle import oracle as orc
    from scipy.special import log_softmax
    cu, cq = orc.make_cfg(w, "fp32"), orc.make_cfg(w, w.dtype)
    lp_g, v_g, v_q = [], [], []
    for n, t in pairs:
        x = gpu["states"][n, t].astype(np.float64)
        a = gpu["actions"][n, t]
        lu = log_softmax(orc.actor(inputs.weights, cu, x))[a]
        vu = orc.critic(inputs.weights, cu, x)
        vq = orc.critic(inputs.weights, cq, x)
        lp_g.append(abs(gpu["logp"][n, t] - lu) / max(abs(lu), 1.0))
        v_g.append(abs(gpu["values"][n, t] - vu) / max(abs(vu), 1.0))
        v_q.append(abs(vq - vu) / max(abs(vu), 1.0))
    v_g, v_q = np.array(v_g), np.array(v_q)
    return {"logp_max": float(max(lp_g)), "value_max": float(v_g.max()), "value_rms": float(np.sqrt((v_g ** 2).mean())),
            "modeq_value_max": float(v_q.max()), "modeq_value_rms": float(np.sqrt((v_q ** 2).mean()))}


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
