"""ctypes wrapper around the C oracle of the PPO update (``oracle/ppo.c``).

TEST INFRASTRUCTURE ONLY: the tests and the benchmark's CPU baseline import
this module; the product path never does.  Everything here is argument
marshalling; the arithmetic is in ``ppo.c``.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading
from dataclasses import dataclass
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ppo.c")
_LIB = os.path.join(_HERE, "_lib", "libppo_oracle.so")
_lock = threading.Lock()
_lib = None


class Shape(C.Structure):
    _fields_ = [("n_market", C.c_int), ("n_actions", C.c_int), ("actor_h1", C.c_int), ("actor_h2", C.c_int),
                ("critic_nh", C.c_int), ("critic_h", C.c_int * 8), ("cur_h", C.c_int)]


class HP(C.Structure):
    _fields_ = [(k, C.c_double) for k in ("clip_eps", "value_coef", "lr", "beta1", "beta2", "adam_eps",
                                            "max_grad_norm", "weight_decay")]


@dataclass
class Hyper:
    """Defaults are the readings stated in the design notes."""
    clip_eps: float = 0.2
    value_coef: float = 1.0
    lr: float = 3e-4
    beta1: float = 0.9
    beta2: float = 0.999
    adam_eps: float = 1e-8
    max_grad_norm: float = 0.5
    weight_decay: float = 0.0

    def c(self) -> HP:
        return HP(*[float(getattr(self, k)) for k, _ in HP._fields_])


def build(force: bool = False) -> str:
    """Compile ``ppo.c`` into ``oracle/_lib/libppo_oracle.so`` (gcc, IEEE double, no contraction)."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(os.path.dirname(_LIB), exist_ok=True)
        tmp = _LIB + f".{os.getpid()}.tmp"
        subprocess.check_call(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                               "-fno-fast-math", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
        return _LIB


def lib():
    global _lib
    if _lib is None:
        L = C.CDLL(build())
        vp = C.c_void_p
        L.ppo_trained_count.restype = C.c_long
        L.ppo_trained_count.argtypes = [C.POINTER(Shape)]
        L.ppo_loss_grad.restype = None
        L.ppo_loss_grad.argtypes = [vp, C.POINTER(Shape), C.POINTER(HP), vp, vp, vp, vp, vp, vp, C.c_int, vp, vp]
        L.ppo_adam_step.restype = C.c_double
        L.ppo_adam_step.argtypes = [vp, vp, vp, vp, C.c_long, C.c_long, C.POINTER(HP)]
        L.ppo_update.restype = C.c_int
        L.ppo_update.argtypes = [vp, C.POINTER(Shape), C.POINTER(HP), vp, vp, vp, vp, vp, vp, C.c_int, C.c_int,
                                 vp, vp, C.POINTER(C.c_long), vp]
        L.ppo_kink_margin.restype = None
        L.ppo_kink_margin.argtypes = [vp, C.POINTER(Shape), vp, vp, C.c_int, vp]
        L.ppo_loss_grad_replay.restype = None
        L.ppo_loss_grad_replay.argtypes = [vp, C.POINTER(Shape), C.POINTER(HP), vp, vp, vp, vp, vp, vp, C.c_int, vp,
                                           vp, vp, C.c_long, C.POINTER(C.c_long), C.POINTER(C.c_long)]
        _lib = L
    return _lib


def shape_of(critic_h=(512, 384, 256, 128, 64)) -> Shape:
    s = Shape()
    s.n_market, s.n_actions, s.actor_h1, s.actor_h2 = 51, 45, 128, 64
    s.critic_nh = len(critic_h)
    for i, h in enumerate(critic_h):
        s.critic_h[i] = h
    s.cur_h = 64
    return s


def _p(a):
    return a.ctypes.data_as(C.c_void_p)


def trained_count(shape: Shape) -> int:
    return int(lib().ppo_trained_count(C.byref(shape)))


@dataclass
class Batch:
    """Tuple arrays of a collection, flattened over (episode, step)."""
    states: np.ndarray    # [T, 54] f32
    actions: np.ndarray   # [T] i32
    logp: np.ndarray      # [T] f32
    adv: np.ndarray       # [T] f32
    ret: np.ndarray       # [T] f32

    def __post_init__(self):
        self.states = np.ascontiguousarray(self.states, dtype=np.float32).reshape(-1, 54)
        self.actions = np.ascontiguousarray(self.actions, dtype=np.int32).reshape(-1)
        self.logp = np.ascontiguousarray(self.logp, dtype=np.float32).reshape(-1)
        self.adv = np.ascontiguousarray(self.adv, dtype=np.float32).reshape(-1)
        self.ret = np.ascontiguousarray(self.ret, dtype=np.float32).reshape(-1)


def loss_grad(params: np.ndarray, shape: Shape, hp: Hyper, b: Batch, rows: np.ndarray):
    """Loss statistics (surrogate, value loss, clipped fraction, mean ratio) and the
    gradient (double, length trained_count) of one mini-batch at double parameters."""
    p = np.ascontiguousarray(params, dtype=np.float64)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    g = np.zeros(trained_count(shape), dtype=np.float64)
    st = np.zeros(4, dtype=np.float64)
    h = hp.c()
    lib().ppo_loss_grad(_p(p), C.byref(shape), C.byref(h), _p(b.states), _p(b.actions), _p(b.logp), _p(b.adv),
                        _p(b.ret), _p(rows), len(rows), _p(g), _p(st))
    return st, g


def loss_grad_replay(params: np.ndarray, shape: Shape, hp: Hyper, b: Batch, rows: np.ndarray, gpu_act: np.ndarray):
    """loss_grad, adopting the path's side of the ReLU kink where its float32
    evaluation may differ from the exact one.  gpu_act: [len(rows), actor hidden |
    critic hidden] float32, the path's hidden activations.  Returns (stats,
    gradient, replays, mismatches)."""
    p = np.ascontiguousarray(params, dtype=np.float64)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    ga = np.ascontiguousarray(gpu_act, dtype=np.float32)
    assert ga.shape[0] == len(rows)
    g = np.zeros(trained_count(shape), dtype=np.float64)
    st = np.zeros(4, dtype=np.float64)
    h = hp.c()
    rep, mis = C.c_long(0), C.c_long(0)
    lib().ppo_loss_grad_replay(_p(p), C.byref(shape), C.byref(h), _p(b.states), _p(b.actions), _p(b.logp), _p(b.adv),
                               _p(b.ret), _p(rows), len(rows), _p(g), _p(st), _p(ga), ga.shape[1], C.byref(rep),
                               C.byref(mis))
    return st, g, rep.value, mis.value


def kink_margin(params: np.ndarray, shape: Shape, b: Batch, rows: np.ndarray) -> np.ndarray:
    """Per row, the smallest relative distance |pre| / (|b| + sum |w x|) of any hidden
    pre-activation from the ReLU kink, at double parameters."""
    p = np.ascontiguousarray(params, dtype=np.float64)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    out = np.zeros(len(rows), dtype=np.float64)
    lib().ppo_kink_margin(_p(p), C.byref(shape), _p(b.states), _p(rows), len(rows), _p(out))
    return out


def adam_step(params: np.ndarray, grad: np.ndarray, m: np.ndarray, v: np.ndarray, t: int, hp: Hyper) -> float:
    """In place on double arrays; returns the gradient norm before clipping."""
    for a in (params, grad, m, v):
        assert a.dtype == np.float64 and a.flags.c_contiguous
    h = hp.c()
    return float(lib().ppo_adam_step(_p(params), _p(grad), _p(m), _p(v), len(params), int(t), C.byref(h)))


class Trainer:
    """The oracle's optimizer state over a packed float32 weight vector."""

    def __init__(self, weights: np.ndarray, critic_h=(512, 384, 256, 128, 64)):
        self.w = np.array(weights, dtype=np.float32)
        self.shape = shape_of(critic_h)
        n = trained_count(self.shape)
        self.m = np.zeros(n, dtype=np.float64)
        self.v = np.zeros(n, dtype=np.float64)
        self.t = C.c_long(0)

    def update(self, b: Batch, rows: np.ndarray, n_steps: int, batch: int, hp: Optional[Hyper] = None):
        """n_steps Adam steps over rows[k*batch:(k+1)*batch]; returns per-step stats [n_steps, 5]."""
        hp = hp or Hyper()
        rows = np.ascontiguousarray(rows, dtype=np.int32)
        assert len(rows) >= n_steps * batch
        st = np.zeros((n_steps, 5), dtype=np.float64)
        h = hp.c()
        rc = lib().ppo_update(_p(self.w), C.byref(self.shape), C.byref(h), _p(b.states), _p(b.actions), _p(b.logp),
                              _p(b.adv), _p(b.ret), _p(rows), int(n_steps), int(batch), _p(self.m), _p(self.v),
                              C.byref(self.t), _p(st))
        if rc != 0:
            raise MemoryError("oracle ppo_update")
        return st
