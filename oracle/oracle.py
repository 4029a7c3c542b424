"""ctypes wrapper around the C oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline import this module; the product path never does.  Everything here is
argument marshalling; the arithmetic is in ``oracle.c``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Dict, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIBDIR = os.path.join(_HERE, "_lib")
_LIB = os.path.join(_LIBDIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

QUANT = {"fp32": 0, "bf16": 1, "tf32": 2}


class OracleCfg(C.Structure):
    _fields_ = [
        ("n_market", C.c_int), ("n_actions", C.c_int), ("actor_h1", C.c_int), ("actor_h2", C.c_int),
        ("critic_nh", C.c_int), ("critic_h", C.c_int * 8), ("cur_h", C.c_int), ("quant", C.c_int),
        ("barrier", C.c_double), ("max_hold", C.c_int), ("pt_scale", C.c_double),
        ("sl_scale", C.c_double), ("div_window", C.c_int), ("div_thresh", C.c_double),
        ("div_penalty", C.c_double), ("cur_coef", C.c_double), ("risk_coef", C.c_double),
        ("tx_base", C.c_double), ("spread", C.c_double),
    ]


class OracleStats(C.Structure):
    _fields_ = [
        ("action_replays", C.c_long), ("done_replays", C.c_long),
        ("action_mismatches", C.c_long), ("done_mismatches", C.c_long),
        ("max_action_gap", C.c_double), ("max_done_gap", C.c_double),
        ("hidden_replays", C.c_long), ("hidden_mismatches", C.c_long), ("max_hidden_excess", C.c_double),
    ]

    def as_dict(self) -> Dict[str, float]:
        return {k: getattr(self, k) for k, _ in self._fields_}


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_lib/liboracle.so`` (gcc, IEEE double, no contraction)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(_LIBDIR, exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = C.CDLL(path)
        p = C.c_void_p
        L.oracle_lcg_step.restype = C.c_uint32
        L.oracle_lcg_step.argtypes = [C.c_uint32]
        L.oracle_lcg_uniform.restype = C.c_double
        L.oracle_lcg_uniform.argtypes = [C.POINTER(C.c_uint32)]
        L.oracle_lcg_fill.restype = None
        L.oracle_lcg_fill.argtypes = [C.c_uint32, C.c_long, C.c_void_p]
        L.oracle_round_bf16.restype = C.c_float
        L.oracle_round_bf16.argtypes = [C.c_float]
        L.oracle_round_tf32.restype = C.c_float
        L.oracle_round_tf32.argtypes = [C.c_float]
        L.oracle_dense.restype = None
        L.oracle_dense.argtypes = [p, p, C.c_int, C.c_int, p, p, C.c_int, C.c_int]
        L.oracle_weight_count.restype = C.c_long
        L.oracle_weight_count.argtypes = [C.POINTER(OracleCfg)]
        L.oracle_actor.restype = None
        L.oracle_actor.argtypes = [p, C.POINTER(OracleCfg), p, p]
        L.oracle_critic.restype = C.c_double
        L.oracle_critic.argtypes = [p, C.POINTER(OracleCfg), p]
        L.oracle_curiosity.restype = None
        L.oracle_curiosity.argtypes = [p, C.POINTER(OracleCfg), p, C.c_int, p]
        L.oracle_sample.restype = C.c_int
        L.oracle_sample.argtypes = [p, C.c_int, C.c_double, p, p]
        L.oracle_exposure.restype = C.c_double
        L.oracle_exposure.argtypes = [C.c_int]
        L.oracle_tx_rate.restype = C.c_double
        L.oracle_tx_rate.argtypes = [C.c_int, C.c_double]
        L.oracle_category.restype = C.c_int
        L.oracle_category.argtypes = [C.c_int]
        L.oracle_window_entropy.restype = C.c_double
        L.oracle_window_entropy.argtypes = [p, C.c_int]
        L.oracle_gae.restype = None
        L.oracle_gae.argtypes = [p, p, p, C.c_int, C.c_double, C.c_double, C.c_double, p, p]
        L.oracle_episode.restype = C.c_int
        L.oracle_rollout.restype = C.c_int
        L.oracle_rollout.argtypes = [p, C.POINTER(OracleCfg), p, C.c_long, p, p, p, C.c_int, C.c_int,
                                     C.c_double, C.c_double, p, p, C.c_double, C.c_double, p, C.c_int,
                                     C.c_double, p, p, p, p, p, p, p, p, p, p, C.POINTER(OracleStats)]
        L.oracle_dense_round_replay.restype = None
        L.oracle_dense_round_replay.argtypes = [p, p, C.c_int, C.c_int, p, p, C.c_int, C.c_int, p,
                                                C.POINTER(OracleStats)]
        L.oracle_hidden_width.restype = C.c_long
        L.oracle_hidden_width.argtypes = [C.POINTER(OracleCfg)]
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(C.c_void_p)


def make_cfg(w, quant: Optional[str] = None) -> OracleCfg:
    """Oracle configuration for a ``workloads.Workload`` (quant defaults to its dtype)."""
    from rl_experience_collection_gb300 import workloads as wl
    c = OracleCfg()
    c.n_market, c.n_actions = wl.N_MARKET, wl.N_ACTIONS
    c.actor_h1, c.actor_h2 = wl.ACTOR_H
    c.critic_nh = len(w.critic_h)
    for i, h in enumerate(w.critic_h):
        c.critic_h[i] = h
    c.cur_h = wl.CUR_H
    c.quant = QUANT[quant if quant is not None else w.dtype]
    c.barrier, c.max_hold = w.barrier, w.max_hold
    c.pt_scale, c.sl_scale = w.pt_scale, w.sl_scale
    c.div_window, c.div_thresh, c.div_penalty = w.div_window, w.div_thresh, w.div_penalty
    c.cur_coef, c.risk_coef, c.tx_base, c.spread = w.cur_coef, w.risk_coef, w.tx_base, w.spread
    return c


# ---------------------------------------------------------------- small calls

def dense_round_replay(W: np.ndarray, b: np.ndarray, x: np.ndarray, relu: bool, quant: int,
                       gpu: Optional[np.ndarray] = None):
    """One layer's rounded outputs under mode Q, replaying the path's rounded
    outputs ``gpu`` where allowed; returns (outputs, stats dict)."""
    W = np.ascontiguousarray(W, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    x = np.ascontiguousarray(x, np.float64)
    g = None if gpu is None else np.ascontiguousarray(gpu, np.float32)
    out = np.zeros(W.shape[0], np.float64)
    st = OracleStats()
    lib().oracle_dense_round_replay(_ptr(W), _ptr(b), W.shape[0], W.shape[1], _ptr(x), _ptr(out), int(relu),
                                    quant, _ptr(g), C.byref(st))
    return out, st.as_dict()


def hidden_width(w) -> int:
    """Floats per row of a path's rounded operands (state input, 64 columns of
    which the first 54 are used | actor h1 | h2 | critic hidden layers |
    curiosity hidden)."""
    return int(lib().oracle_hidden_width(C.byref(make_cfg(w))))


def lcg_step(s: int) -> int:
    return lib().oracle_lcg_step(s)


def lcg_uniforms(seed: int, n: int) -> np.ndarray:
    out = np.zeros(n, np.float64)
    lib().oracle_lcg_fill(seed, n, _ptr(out))
    return out


def round_bf16(x: float) -> float:
    return lib().oracle_round_bf16(x)


def round_tf32(x: float) -> float:
    return lib().oracle_round_tf32(x)


def dense(W: np.ndarray, b: np.ndarray, x: np.ndarray, relu: bool, quant: int = 0) -> np.ndarray:
    W = np.ascontiguousarray(W, np.float32)
    b = np.ascontiguousarray(b, np.float32)
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros(W.shape[0], np.float64)
    lib().oracle_dense(_ptr(W), _ptr(b), W.shape[0], W.shape[1], _ptr(x), _ptr(out), int(relu), quant)
    return out


def actor(weights: np.ndarray, cfg: OracleCfg, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros(cfg.n_actions, np.float64)
    lib().oracle_actor(_ptr(weights), C.byref(cfg), _ptr(x), _ptr(out))
    return out


def critic(weights: np.ndarray, cfg: OracleCfg, x: np.ndarray) -> float:
    x = np.ascontiguousarray(x, np.float64)
    return lib().oracle_critic(_ptr(weights), C.byref(cfg), _ptr(x))


def curiosity(weights: np.ndarray, cfg: OracleCfg, x: np.ndarray, a: int) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    out = np.zeros(cfg.n_market + 3, np.float64)
    lib().oracle_curiosity(_ptr(weights), C.byref(cfg), _ptr(x), int(a), _ptr(out))
    return out


def sample(logits: np.ndarray, u: float):
    """(action, log p[action], cdf) for one draw."""
    l = np.ascontiguousarray(logits, np.float64)
    cdf = np.zeros(l.size, np.float64)
    lp = C.c_double()
    a = lib().oracle_sample(_ptr(l), l.size, u, C.byref(lp), _ptr(cdf))
    return a, lp.value, cdf


def exposure(a: int) -> float:
    return lib().oracle_exposure(a)


def tx_rate(a: int, base: float) -> float:
    return lib().oracle_tx_rate(a, base)


def category(a: int) -> int:
    return lib().oracle_category(a)


def window_entropy(cats: Sequence[int]) -> float:
    arr = np.ascontiguousarray(cats, np.int32)
    return lib().oracle_window_entropy(_ptr(arr), arr.size)


def gae(r, v, d, v_boot: float, gamma: float, lam: float):
    r = np.ascontiguousarray(r, np.float64)
    v = np.ascontiguousarray(v, np.float64)
    d = np.ascontiguousarray(d, np.int32)
    adv = np.zeros(r.size)
    ret = np.zeros(r.size)
    lib().oracle_gae(_ptr(r), _ptr(v), _ptr(d), r.size, v_boot, gamma, lam, _ptr(adv), _ptr(ret))
    return adv, ret


# ---------------------------------------------------------------- rollouts

def rollout(w, inputs, idx: Sequence[int], quant: Optional[str] = None, horizon: Optional[int] = None,
            gpu_actions: Optional[np.ndarray] = None, gpu_dones: Optional[np.ndarray] = None,
            act_band: float = 1e-5, done_band: float = 1e-6, threads: int = 1,
            gamma: Optional[float] = None, lam: Optional[float] = None,
            gpu_hidden: Optional[np.ndarray] = None, return_hidden: bool = False, state_band: float = 2e-6):
    """Oracle outputs for episodes ``idx`` of a batch.

    ``gpu_hidden`` (optional, float32 ``[n_h, L + 1, hidden_width(w)]``): the
    path under test's rounded operands of episodes ``0..n_h-1`` (row t per
    step, row L the bootstrap critic: state input, actor h1, h2, critic
    hidden layers, curiosity hidden), replayed under mode Q where they differ
    from the oracle's own rounding within the float32 accumulation bound (the
    state input within ``state_band`` relative to max(|x|, 1)); counted in
    ``stats``: ``hidden_replays``, and ``hidden_mismatches`` for any other
    difference.  ``return_hidden``:
    also return the hidden activations the oracle used, as ``hidden``
    ([len(idx), L + 1, hidden_width(w)]).
    Returns a dict of arrays with a leading axis ``len(idx)`` plus ``stats``.
    ``threads > 1`` runs disjoint episode subsets on Python threads (the C
    call releases the GIL); the arithmetic is unchanged.
    """
    L = w.horizon if horizon is None else horizon
    g = w.gamma if gamma is None else gamma
    lm = w.lam if lam is None else lam
    cfg = make_cfg(w, quant)
    idx = np.ascontiguousarray(idx, np.int32)
    n = idx.size
    sd = cfg.n_market + 3
    out = {
        "states": np.zeros((n, L, sd), np.float32), "actions": np.zeros((n, L), np.int32),
        "logp": np.zeros((n, L), np.float32), "values": np.zeros((n, L), np.float32),
        "rewards": np.zeros((n, L), np.float32), "dones": np.zeros((n, L), np.int32),
        "adv": np.zeros((n, L), np.float32), "ret": np.zeros((n, L), np.float32),
        "vboot": np.zeros(n, np.float64),
    }
    if return_hidden:
        out["hidden"] = np.zeros((n, L + 1, hidden_width(w)), np.float32)
    feats = np.ascontiguousarray(inputs.features, np.float32)
    starts = np.ascontiguousarray(inputs.starts, np.int32)
    seeds = np.ascontiguousarray(inputs.seeds, np.uint32)
    weights = np.ascontiguousarray(inputs.weights, np.float32)
    gh = None if gpu_hidden is None else np.ascontiguousarray(gpu_hidden, np.float32)
    n_h = 0 if gh is None else gh.shape[0]
    if gh is not None and gh.shape[1:] != (L + 1, hidden_width(w)):
        raise ValueError(f"gpu_hidden has shape {gh.shape}, want [n, {L + 1}, {hidden_width(w)}]")
    ga = None if gpu_actions is None else np.ascontiguousarray(gpu_actions, np.int32)
    gd = None if gpu_dones is None else np.ascontiguousarray(gpu_dones, np.int32)
    L_ = lib()

    def run(lo: int, hi: int) -> OracleStats:
        st = OracleStats()
        sub = idx[lo:hi]
        rc = L_.oracle_rollout(
            _ptr(weights), C.byref(cfg), _ptr(feats), feats.shape[0], _ptr(starts), _ptr(seeds),
            _ptr(sub), sub.size, L, g, lm, _ptr(ga), _ptr(gd), act_band, done_band, _ptr(gh), n_h, state_band,
            _ptr(out["hidden"][lo:hi]) if return_hidden else None,
            _ptr(out["states"][lo:hi]), _ptr(out["actions"][lo:hi]), _ptr(out["logp"][lo:hi]),
            _ptr(out["values"][lo:hi]), _ptr(out["rewards"][lo:hi]), _ptr(out["dones"][lo:hi]),
            _ptr(out["adv"][lo:hi]), _ptr(out["ret"][lo:hi]), _ptr(out["vboot"][lo:hi]), C.byref(st))
        if rc != 0:
            raise ValueError(f"oracle_rollout rejected its arguments (rc={rc})")
        return st

    if threads <= 1 or n <= 1:
        stats = [run(0, n)]
    else:
        bounds = np.linspace(0, n, min(threads, n) + 1).astype(int)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            stats = list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    tot = {k: 0 for k, _ in OracleStats._fields_}
    for s in stats:
        d = s.as_dict()
        for k in tot:
            tot[k] = max(tot[k], d[k]) if k.startswith("max_") else tot[k] + d[k]
    out["stats"] = tot
    return out
