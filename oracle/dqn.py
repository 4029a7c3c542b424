"""ctypes wrapper around the C oracle of DQN experience collection (``oracle/dqn.c``,
which includes ``oracle/oracle.c`` for the shared environment).

TEST INFRASTRUCTURE ONLY: the tests and the smoke check import this module;
the product path never does.  Everything here is argument marshalling; the arithmetic is in the C files.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor
from typing import Optional, Sequence

import numpy as np

from . import oracle as orc

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "dqn.c"), os.path.join(_HERE, "oracle.c")]
_LIB = os.path.join(_HERE, "_lib", "libdqn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``dqn.c`` (with ``oracle.c``) into ``oracle/_lib/libdqn_oracle.so``."""
    with _lock:
        newest = max(os.path.getmtime(p) for p in _SRCS)
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= newest:
            return _LIB
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-I", _HERE, "-o", tmp, _SRCS[0], "-lm"])
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        p = C.c_void_p
        cfg = C.POINTER(orc.OracleCfg)
        L.dqn_net_count.restype = C.c_long
        L.dqn_net_count.argtypes = [cfg]
        L.dqn_q_parts.restype = None
        L.dqn_q_parts.argtypes = [p, cfg, p, p, p]
        L.dqn_q.restype = None
        L.dqn_q.argtypes = [p, cfg, p, p]
        L.dqn_rollout.restype = C.c_int
        L.dqn_rollout.argtypes = [p, cfg, p, C.c_long, p, p, p, C.c_int, C.c_int, C.c_double, C.c_double,
                                  C.c_int, p, p, C.c_double, C.c_double, p, p, p, p, p, p, p, p,
                                  C.POINTER(orc.OracleStats)]
        _lib = L
    return _lib


_ptr = orc._ptr


def net_count(cfg) -> int:
    return lib().dqn_net_count(C.byref(cfg))


def q_parts(net: np.ndarray, cfg, x: np.ndarray):
    """(V, A[45]) of state x under one net."""
    x = np.ascontiguousarray(x, np.float64)
    v = np.zeros(1)
    a = np.zeros(cfg.n_actions)
    lib().dqn_q_parts(_ptr(np.ascontiguousarray(net, np.float32)), C.byref(cfg), _ptr(x), _ptr(v), _ptr(a))
    return v[0], a


def q_values(net: np.ndarray, cfg, x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float64)
    q = np.zeros(cfg.n_actions)
    lib().dqn_q(_ptr(np.ascontiguousarray(net, np.float32)), C.byref(cfg), _ptr(x), _ptr(q))
    return q


def rollout(w, inputs, weights: np.ndarray, idx: Sequence[int], epsilon: float, quant: Optional[str] = None,
            horizon: Optional[int] = None, gamma: Optional[float] = None, gpu_actions=None, gpu_dones=None,
            q_band: float = 0.0, done_band: float = 1e-6, threads: int = 1, recycle: bool = False):
    """Oracle outputs (states, next_states, actions, rewards, dones, q, td, bars;
    leading axis len(idx)) of the DQN collector for episodes idx, plus ``stats``.
    recycle: after a done, the next step starts at a fresh bar from the LCG."""
    L = w.horizon if horizon is None else horizon
    g = w.gamma if gamma is None else gamma
    cfg = orc.make_cfg(w, quant)
    idx = np.ascontiguousarray(idx, np.int32)
    n, sd = idx.size, cfg.n_market + 3
    out = {"states": np.zeros((n, L, sd), np.float32), "next_states": np.zeros((n, L, sd), np.float32),
           "actions": np.zeros((n, L), np.int32), "rewards": np.zeros((n, L), np.float32),
           "dones": np.zeros((n, L), np.int32), "q": np.zeros((n, L), np.float32),
           "td": np.zeros((n, L), np.float32), "bars": np.zeros((n, L), np.int32)}
    feats = np.ascontiguousarray(inputs.features, np.float32)
    starts = np.ascontiguousarray(inputs.starts, np.int32)
    seeds = np.ascontiguousarray(inputs.seeds, np.uint32)
    wts = np.ascontiguousarray(weights, np.float32)
    ga = None if gpu_actions is None else np.ascontiguousarray(gpu_actions, np.int32)
    gd = None if gpu_dones is None else np.ascontiguousarray(gpu_dones, np.int32)
    L_ = lib()

    def run(lo, hi):
        st = orc.OracleStats()
        sub = idx[lo:hi]
        rc = L_.dqn_rollout(_ptr(wts), C.byref(cfg), _ptr(feats), feats.shape[0], _ptr(starts), _ptr(seeds),
                            _ptr(sub), sub.size, L, g, float(np.float32(epsilon)), int(recycle), _ptr(ga),
                            _ptr(gd), q_band, done_band, _ptr(out["states"][lo:hi]), _ptr(out["actions"][lo:hi]),
                            _ptr(out["rewards"][lo:hi]), _ptr(out["dones"][lo:hi]), _ptr(out["q"][lo:hi]),
                            _ptr(out["td"][lo:hi]), _ptr(out["next_states"][lo:hi]), _ptr(out["bars"][lo:hi]),
                            C.byref(st))
        if rc != 0:
            raise ValueError(f"dqn_rollout rejected its arguments (rc={rc})")
        return st

    if threads <= 1 or n <= 1:
        stats = [run(0, n)]
    else:
        bounds = np.linspace(0, n, min(threads, n) + 1).astype(int)
        with ThreadPoolExecutor(len(bounds) - 1) as ex:
            stats = list(ex.map(lambda i: run(bounds[i], bounds[i + 1]), range(len(bounds) - 1)))
    tot = {k: 0 for k, _ in orc.OracleStats._fields_}
    for s in stats:
        d = s.as_dict()
        for k in tot:
            tot[k] = max(tot[k], d[k]) if k.startswith("max_") else tot[k] + d[k]
    out["stats"] = tot
    return out
