"""Thin Python binding of the C ABI in ``include/rollout.h`` (ctypes).

Argument marshalling only: every step of the computation runs in
``librollout.so``.  There is no fallback -- if the library is missing or fails
to load, :func:`lib` raises.  PyTorch supplies device memory and streams.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import Dict, Optional

from . import workloads as wl

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "librollout.so")

ROLLOUT_OK = 0
ROLLOUT_ERR_INVALID = -1
ROLLOUT_ERR_RANGE = -2
ROLLOUT_ERR_CUDA = -3
ROLLOUT_ERR_TIMEOUT = -4
ROLLOUT_ERR_UNSUPPORTED = -5
ROLLOUT_ERR_NOMEM = -6
DTYPE = {"fp32": 0, "tf32": 1, "bf16": 2}

EXPORTS = ["rollout_create", "rollout_set_weights", "rollout_run", "rollout_status", "rollout_destroy",
           "rollout_last_error", "rollout_set_timing", "rollout_phase_ms", "rollout_run_static", "rollout_run_host",
           "rollout_set_weights_device", "rollout_test_stall", "rollout_test_activations",
           "rollout_test_alloc", "rollout_forward"]


class RolloutDims(C.Structure):
    _fields_ = [
        ("n_market", C.c_int), ("n_actions", C.c_int), ("actor_h1", C.c_int), ("actor_h2", C.c_int),
        ("critic_nh", C.c_int), ("critic_h", C.c_int * 8), ("cur_h", C.c_int), ("dtype", C.c_int),
        ("n_bars", C.c_int), ("barrier", C.c_float), ("max_hold", C.c_int), ("pt_scale", C.c_float),
        ("sl_scale", C.c_float), ("div_window", C.c_int), ("div_thresh", C.c_float),
        ("div_penalty", C.c_float), ("cur_coef", C.c_float), ("risk_coef", C.c_float),
        ("tx_base", C.c_float), ("spread", C.c_float),
    ]


PPO_EXPORTS = ["ppo_create", "ppo_update", "ppo_gradient", "ppo_get_weights", "ppo_reset_optimizer", "ppo_status",
               "ppo_device_weights", "ppo_test_activations",
               "ppo_destroy"]


class PpoHparams(C.Structure):
    """include/ppo.h ppo_hparams; defaults are the readings stated in the design notes."""
    _fields_ = [(k, C.c_float) for k in ("clip_eps", "value_coef", "lr", "beta1", "beta2", "adam_eps",
                                           "max_grad_norm", "weight_decay")]

    @classmethod
    def make(cls, clip_eps=0.2, value_coef=1.0, lr=3e-4, beta1=0.9, beta2=0.999, adam_eps=1e-8, max_grad_norm=0.5,
             weight_decay=0.0):
        return cls(clip_eps, value_coef, lr, beta1, beta2, adam_eps, max_grad_norm, weight_decay)


PER_EXPORTS = ["per_create", "per_insert", "per_sample", "per_update_priorities", "per_size", "per_read",
               "per_status", "per_destroy"]


DQN_EXPORTS = ["dqn_weight_count", "dqn_create", "dqn_set_weights", "dqn_run", "dqn_status", "dqn_destroy",
               "dqn_set_timing", "dqn_phase_ms", "dqn_test_stall", "dqn_set_recycle"]
DQN_OUTPUTS = ("states", "actions", "rewards", "dones", "q", "td", "next_states")


class RolloutError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"rollout error {code}: {msg}")
        self.code = code


_lib = None


def lib(path: Optional[str] = None):
    """Loads librollout.so (raises if it is missing: there is no fallback path)."""
    global _lib
    if _lib is not None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"{p} is missing: build it with rl_experience_collection_gb300.build.build() "
                           "(there is no CPU fallback)")
    L = C.CDLL(p)
    vp = C.c_void_p
    L.rollout_create.restype = C.c_int
    L.rollout_create.argtypes = [vp, C.POINTER(RolloutDims), C.POINTER(vp)]
    L.rollout_set_weights.restype = C.c_int
    L.rollout_set_weights.argtypes = [vp, vp]
    L.rollout_set_weights_device.restype = C.c_int
    L.rollout_set_weights_device.argtypes = [vp, vp, vp]
    L.rollout_run.restype = C.c_int
    L.rollout_run.argtypes = [vp, vp, vp, vp, C.c_int, C.c_int, C.c_float, C.c_float,
                              vp, vp, vp, vp, vp, vp, vp, vp, vp]
    L.rollout_run_static.restype = C.c_int
    L.rollout_run_static.argtypes = list(L.rollout_run.argtypes)
    L.rollout_run_host.restype = C.c_int
    L.rollout_run_host.argtypes = list(L.rollout_run.argtypes)
    L.rollout_status.restype = C.c_int
    L.rollout_status.argtypes = [vp]
    L.rollout_destroy.restype = None
    L.rollout_destroy.argtypes = [vp]
    L.rollout_set_timing.restype = C.c_int
    L.rollout_set_timing.argtypes = [vp, C.c_int]
    L.rollout_phase_ms.restype = C.c_int
    L.rollout_phase_ms.argtypes = [vp, C.POINTER(C.c_float)]
    L.rollout_test_stall.restype = C.c_int
    L.rollout_test_stall.argtypes = [vp, C.c_int]
    L.rollout_test_activations.restype = C.c_int
    L.rollout_test_activations.argtypes = [vp, vp, C.c_int]
    L.rollout_forward.restype = C.c_int
    L.rollout_forward.argtypes = [vp, vp, vp, C.c_int, vp, vp, vp, vp]
    L.rollout_test_alloc.restype = C.c_int
    L.rollout_test_alloc.argtypes = [C.c_longlong, C.POINTER(C.c_longlong)]
    L.rollout_last_error.restype = C.c_char_p
    L.rollout_last_error.argtypes = []
    L.dqn_weight_count.restype = C.c_longlong
    L.dqn_weight_count.argtypes = []
    L.dqn_create.restype = C.c_int
    L.dqn_create.argtypes = [vp, C.POINTER(RolloutDims), C.POINTER(vp)]
    L.dqn_set_weights.restype = C.c_int
    L.dqn_set_weights.argtypes = [vp, vp]
    L.dqn_run.restype = C.c_int
    L.dqn_run.argtypes = [vp, vp, vp, vp, C.c_int, C.c_int, C.c_float, C.c_float, vp, vp, vp, vp, vp, vp, vp, vp]
    L.dqn_status.restype = C.c_int
    L.dqn_status.argtypes = [vp]
    L.dqn_set_timing.restype = C.c_int
    L.dqn_set_timing.argtypes = [vp, C.c_int]
    L.dqn_phase_ms.restype = C.c_int
    L.dqn_phase_ms.argtypes = [vp, C.POINTER(C.c_float)]
    L.dqn_test_stall.restype = C.c_int
    L.dqn_test_stall.argtypes = [vp, C.c_int]
    L.dqn_set_recycle.restype = C.c_int
    L.dqn_set_recycle.argtypes = [vp, C.c_int]
    L.dqn_destroy.restype = None
    L.dqn_destroy.argtypes = [vp]
    L.per_create.restype = C.c_int
    L.per_create.argtypes = [C.c_longlong, C.c_int, C.POINTER(vp)]
    L.per_insert.restype = C.c_int
    L.per_insert.argtypes = [vp, vp, vp, vp, vp, vp, C.c_longlong, vp]
    L.per_sample.restype = C.c_int
    L.per_sample.argtypes = [vp, C.c_int, C.c_float, C.c_uint64, C.c_uint64, vp, vp, vp, vp, vp, vp, vp, vp]
    L.per_update_priorities.restype = C.c_int
    L.per_update_priorities.argtypes = [vp, vp, vp, C.c_int, C.c_float, C.c_float, vp]
    L.per_size.restype = C.c_int
    L.per_size.argtypes = [vp, C.POINTER(C.c_longlong), C.POINTER(C.c_longlong)]
    L.per_read.restype = C.c_int
    L.per_read.argtypes = [vp, vp, vp, vp]
    L.per_status.restype = C.c_int
    L.per_status.argtypes = [vp]
    L.per_destroy.restype = None
    L.per_destroy.argtypes = [vp]
    L.ppo_device_weights.restype = C.c_int
    L.ppo_device_weights.argtypes = [vp, C.POINTER(vp)]
    L.ppo_create.restype = C.c_int
    L.ppo_create.argtypes = [vp, C.POINTER(RolloutDims), C.POINTER(vp)]
    L.ppo_update.restype = C.c_int
    L.ppo_update.argtypes = [vp, vp, vp, vp, vp, vp, C.c_longlong, vp, C.c_int, C.c_int, C.POINTER(PpoHparams),
                             vp, vp]
    L.ppo_gradient.restype = C.c_int
    L.ppo_gradient.argtypes = [vp, vp, vp, vp, vp, vp, C.c_longlong, vp, C.c_int, C.POINTER(PpoHparams), vp, vp, vp]
    L.ppo_get_weights.restype = C.c_int
    L.ppo_get_weights.argtypes = [vp, vp, vp]
    L.ppo_test_activations.restype = C.c_int
    L.ppo_test_activations.argtypes = [vp, vp, vp]
    L.ppo_reset_optimizer.restype = C.c_int
    L.ppo_reset_optimizer.argtypes = [vp, vp]
    L.ppo_status.restype = C.c_int
    L.ppo_status.argtypes = [vp]
    L.ppo_destroy.restype = None
    L.ppo_destroy.argtypes = [vp]
    _lib = L
    return L


def test_alloc(fail_at: int = 0) -> int:
    """Test hook: the fail_at-th device allocation of rollout handles from now on
    fails as out of memory (0: none).  Returns the live allocations."""
    live = C.c_longlong()
    _check(lib().rollout_test_alloc(int(fail_at), C.byref(live)))
    return live.value


def last_error() -> str:
    return lib().rollout_last_error().decode()


def _check(rc: int):
    if rc != ROLLOUT_OK:
        raise RolloutError(rc, last_error())


def make_dims(w: wl.Workload, n_bars: Optional[int] = None, dtype: Optional[str] = None) -> RolloutDims:
    d = RolloutDims()
    d.n_market, d.n_actions = wl.N_MARKET, wl.N_ACTIONS
    d.actor_h1, d.actor_h2 = wl.ACTOR_H
    d.critic_nh = len(w.critic_h)
    for i, h in enumerate(w.critic_h):
        d.critic_h[i] = h
    d.cur_h = wl.CUR_H
    d.dtype = DTYPE[dtype or w.dtype]
    d.n_bars = w.n_bars if n_bars is None else n_bars
    d.barrier, d.max_hold = w.barrier, w.max_hold
    d.pt_scale, d.sl_scale = w.pt_scale, w.sl_scale
    d.div_window, d.div_thresh, d.div_penalty = w.div_window, w.div_thresh, w.div_penalty
    d.cur_coef, d.risk_coef, d.tx_base, d.spread = w.cur_coef, w.risk_coef, w.tx_base, w.spread
    return d


OUTPUTS = ("states", "actions", "logp", "values", "rewards", "dones", "adv", "ret")


def make_outputs(N: int, L: int, device="cuda") -> Dict[str, "torch.Tensor"]:
    import torch
    f32, i32 = torch.float32, torch.int32
    return {
        "states": torch.empty((N, L, wl.STATE_DIM), dtype=f32, device=device),
        "actions": torch.empty((N, L), dtype=i32, device=device),
        "logp": torch.empty((N, L), dtype=f32, device=device),
        "values": torch.empty((N, L), dtype=f32, device=device),
        "rewards": torch.empty((N, L), dtype=f32, device=device),
        "dones": torch.empty((N, L), dtype=i32, device=device),
        "adv": torch.empty((N, L), dtype=f32, device=device),
        "ret": torch.empty((N, L), dtype=f32, device=device),
    }


class Rollout:
    """Owns a ``rollout_handle``: ``rollout_create`` on construction, ``rollout_destroy`` on close."""

    def __init__(self, weights, dims: RolloutDims):
        import numpy as np
        self._w = np.ascontiguousarray(weights, dtype=np.float32)
        self.dims = dims
        h = C.c_void_p()
        _check(lib().rollout_create(self._w.ctypes.data_as(C.c_void_p), C.byref(dims), C.byref(h)))
        self._h = h

    @classmethod
    def for_workload(cls, w: wl.Workload, weights, n_bars: Optional[int] = None, dtype: Optional[str] = None):
        return cls(weights, make_dims(w, n_bars, dtype))

    def set_weights(self, weights):
        import numpy as np
        self._w = np.ascontiguousarray(weights, dtype=np.float32)
        _check(lib().rollout_set_weights(self._h, self._w.ctypes.data_as(C.c_void_p)))

    def set_weights_device(self, weights, stream=None) -> None:
        """rollout_set_weights_device: enqueues the refresh from a contiguous float32
        CUDA tensor of the packed weights, or a device address of them (for example
        PpoTrainer.device_weights())."""
        if isinstance(weights, int):
            ptr = weights
        elif weights.is_cuda and weights.is_contiguous() and weights.dtype.itemsize == 4:
            ptr = weights.data_ptr()
        else:
            raise ValueError("weights must be a contiguous float32 CUDA tensor or a device address")
        _check(lib().rollout_set_weights_device(self._h, C.c_void_p(ptr), C.c_void_p(_stream_handle(stream))))

    def run(self, features, starts, seeds, N: int, L: int, gamma: float, lam: float,
            out: Dict[str, "torch.Tensor"], stream=None) -> None:
        """Enqueues one collection on ``stream`` (a torch.cuda.Stream, a raw handle, or None = current)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        p = lambda t: C.c_void_p(t.data_ptr())
        _check(lib().rollout_run(self._h, p(features), p(starts), p(seeds), int(N), int(L), float(gamma),
                                 float(lam), p(out["states"]), p(out["actions"]), p(out["logp"]),
                                 p(out["values"]), p(out["rewards"]), p(out["dones"]), p(out["adv"]),
                                 p(out["ret"]), C.c_void_p(sh)))

    def run_static(self, features, starts, seeds, N: int, L: int, gamma: float, lam: float,
                   out: Dict[str, "torch.Tensor"], stream=None) -> None:
        """rollout_run_static: same as run(), with the value phase's scratch taken
        from the library's fixed device array instead of handle-owned memory."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
        p = lambda t: C.c_void_p(t.data_ptr())
        _check(lib().rollout_run_static(self._h, p(features), p(starts), p(seeds), int(N), int(L), float(gamma),
                                        float(lam), p(out["states"]), p(out["actions"]), p(out["logp"]),
                                        p(out["values"]), p(out["rewards"]), p(out["dones"]), p(out["adv"]),
                                        p(out["ret"]), C.c_void_p(sh)))

    def run_host(self, features, starts, seeds, N: int, L: int, gamma: float, lam: float,
                 out: Dict[str, object], stream=None) -> None:
        """rollout_run_host: inputs and outputs in HOST memory (numpy arrays or CPU
        tensors, page-locked for the copies to overlap the kernels).  `out` maps
        output names (OUTPUTS) to host arrays; a missing name is not copied back.
        Enqueues on `stream` (a torch.cuda.Stream, a raw handle, or None = current)."""
        import torch
        if stream is None:
            stream = torch.cuda.current_stream()
        sh = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)

        def p(x):
            if x is None:
                return C.c_void_p(None)
            return C.c_void_p(x.data_ptr() if hasattr(x, "data_ptr") else x.ctypes.data)

        o = [out.get(k) for k in ("states", "actions", "logp", "values", "rewards", "dones", "adv", "ret")]
        _check(lib().rollout_run_host(self._h, p(features), p(starts), p(seeds), int(N), int(L), float(gamma),
                                      float(lam), *[p(x) for x in o], C.c_void_p(sh)))

    def run_raw(self, ptrs, N: int, L: int, gamma: float, lam: float, stream_handle: int = 0) -> int:
        """Raw-pointer form (integers), returns the status code instead of raising."""
        return lib().rollout_run(self._h, *[C.c_void_p(x) for x in ptrs[:3]], int(N), int(L), float(gamma),
                                 float(lam), *[C.c_void_p(x) for x in ptrs[3:]], C.c_void_p(stream_handle))

    def set_timing(self, on: bool = True) -> None:
        _check(lib().rollout_set_timing(self._h, int(on)))

    def phase_ms(self):
        """Device milliseconds of the last run's rollout, state-row, value and GAE kernels."""
        ms = (C.c_float * 4)()
        _check(lib().rollout_phase_ms(self._h, ms))
        return [float(x) for x in ms]

    def test_stall(self, on: bool = True) -> None:
        """Test hook: later runs launch the value kernel's stalling test build."""
        _check(lib().rollout_test_stall(self._h, int(on)))

    def forward(self, states, actions, stream=None):
        """rollout_forward: (logits [M, 45], values [M], cur_pred [M, 54]) of the
        device tensors states [M, 54] float32 and actions [M] int32."""
        import torch
        M = int(states.shape[0])
        dev = states.device
        logits = torch.empty((M, wl.N_ACTIONS), dtype=torch.float32, device=dev)
        values = torch.empty(M, dtype=torch.float32, device=dev)
        cur = torch.empty((M, wl.STATE_DIM), dtype=torch.float32, device=dev)
        st = states.contiguous()
        ac = actions.contiguous()
        _check(lib().rollout_forward(self._h, C.c_void_p(st.data_ptr()), C.c_void_p(ac.data_ptr()), M,
                                     C.c_void_p(logits.data_ptr()), C.c_void_p(values.data_ptr()),
                                     C.c_void_p(cur.data_ptr()), C.c_void_p(_stream_handle(stream))))
        return logits, values, cur

    def test_activations(self, dump=None, n_episodes: int = 0) -> None:
        """Test hook: later runs also write the rounded hidden activations of
        episodes 0..n_episodes-1 into the device tensor ``dump``
        ([n_episodes, L + 1, activation_width] float32); None turns it off."""
        ptr = None if dump is None else dump.data_ptr()
        self._dump = dump                        # keeps the array alive while runs may use it
        _check(lib().rollout_test_activations(self._h, ptr, int(n_episodes) if dump is not None else 0))

    def status(self) -> int:
        return lib().rollout_status(self._h)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().rollout_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class PpoTrainer:
    """Owns a ``ppo_trainer`` (include/ppo.h): a float32 device copy of the packed
    weights and its Adam state."""

    def __init__(self, weights, dims: RolloutDims):
        import numpy as np
        self._w = np.ascontiguousarray(weights, dtype=np.float32)
        h = C.c_void_p()
        _check(lib().ppo_create(self._w.ctypes.data_as(C.c_void_p), C.byref(dims), C.byref(h)))
        self._h = h
        self.n_weights = self._w.size
        self.critic_h = tuple(dims.critic_h[i] for i in range(dims.critic_nh))

    @classmethod
    def for_workload(cls, w: wl.Workload, weights):
        return cls(weights, make_dims(w))

    def update(self, states, actions, logp_old, adv, ret, indices, n_steps: int, batch: int,
               hp: Optional[PpoHparams] = None, stats=None, stream=None) -> None:
        """Enqueues n_steps Adam steps; all arrays are device tensors (tuples flattened
        over episode and step; indices int32, n_steps*batch of them)."""
        hp = hp or PpoHparams.make()
        T = actions.numel()
        p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(None)
        _check(lib().ppo_update(self._h, p(states), p(actions), p(logp_old), p(adv), p(ret), int(T), p(indices),
                                int(n_steps), int(batch), C.byref(hp), p(stats), C.c_void_p(_stream_handle(stream))))

    def gradient(self, states, actions, logp_old, adv, ret, indices, batch: int, grad, stats=None,
                 hp: Optional[PpoHparams] = None, stream=None) -> None:
        """Enqueues the loss statistics and gradient of one mini-batch at the current
        weights (grad: a device float32 tensor of the actor + critic parameter count)."""
        hp = hp or PpoHparams.make()
        T = actions.numel()
        p = lambda t: C.c_void_p(t.data_ptr()) if t is not None else C.c_void_p(None)
        _check(lib().ppo_gradient(self._h, p(states), p(actions), p(logp_old), p(adv), p(ret), int(T), p(indices),
                                  int(batch), C.byref(hp), p(grad), p(stats), C.c_void_p(_stream_handle(stream))))

    def weights(self, stream=None):
        """The packed float32 weights, as a host numpy array (synchronises the stream)."""
        import numpy as np
        import torch
        out = np.empty(self.n_weights, dtype=np.float32)
        _check(lib().ppo_get_weights(self._h, out.ctypes.data_as(C.c_void_p), C.c_void_p(_stream_handle(stream))))
        torch.cuda.synchronize()
        return out

    def weights_into(self, out, stream=None) -> None:
        """Enqueues a device-to-device copy of the packed float32 weights into `out`
        (a contiguous float32 CUDA tensor of n_weights elements); no synchronisation."""
        if not (out.is_cuda and out.is_contiguous()) or out.numel() != self.n_weights or out.dtype.itemsize != 4:
            raise ValueError("out must be a contiguous float32 CUDA tensor of n_weights elements")
        _check(lib().ppo_get_weights(self._h, C.c_void_p(out.data_ptr()), C.c_void_p(_stream_handle(stream))))

    def activations(self, batch: int, stream=None):
        """Test hook: the last forward pass's hidden activations, [batch, actor
        hidden | critic hidden] float32 (numpy, after a synchronise)."""
        import numpy as np
        import torch
        width = wl.ACTOR_H[0] + wl.ACTOR_H[1] + int(sum(self.critic_h))
        out = torch.empty((batch, width), dtype=torch.float32, device="cuda")
        _check(lib().ppo_test_activations(self._h, C.c_void_p(out.data_ptr()), C.c_void_p(_stream_handle(stream))))
        torch.cuda.synchronize()
        return out.cpu().numpy()

    def device_weights(self) -> int:
        """ppo_device_weights: the address of the trainer's own device weights (updated
        in place by update()), for Rollout.set_weights_device."""
        p = C.c_void_p()
        _check(lib().ppo_device_weights(self._h, C.byref(p)))
        return p.value

    def reset_optimizer(self, stream=None) -> None:
        _check(lib().ppo_reset_optimizer(self._h, C.c_void_p(_stream_handle(stream))))

    def status(self) -> int:
        return lib().ppo_status(self._h)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().ppo_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


DUMP_IN_COLS = 64


def activation_width(critic_h) -> int:
    """Floats per row of rollout_test_activations' array: state input (64
    columns, the first 54 used) | actor h1 | h2 | critic hidden layers |
    curiosity hidden."""
    return DUMP_IN_COLS + wl.ACTOR_H[0] + wl.ACTOR_H[1] + int(sum(critic_h)) + wl.CUR_H


def collect(w: wl.Workload, inputs: "wl.Inputs", N: Optional[int] = None, L: Optional[int] = None,
            device="cuda", handle: Optional[Rollout] = None, dump_episodes: int = 0) -> Dict[str, "torch.Tensor"]:
    """One-call convenience: uploads inputs, runs one collection, returns device outputs.
    dump_episodes > 0 (tf32 / bf16 only) also returns, under "hidden", the rounded
    hidden activations of episodes 0..dump_episodes-1 (rollout_test_activations)."""
    import torch
    N = w.n_episodes if N is None else N
    L = w.horizon if L is None else L
    h = handle or Rollout.for_workload(w, inputs.weights, n_bars=inputs.features.shape[0])
    feats = torch.from_numpy(inputs.features).to(device)
    starts = torch.from_numpy(inputs.starts[:N]).to(device)
    seeds = torch.from_numpy(inputs.seeds[:N].view("int32")).to(device)
    out = make_outputs(N, L, device)
    dump = None
    if dump_episodes > 0:
        k = min(dump_episodes, N)
        dump = torch.full((k, L + 1, activation_width(w.critic_h)), float("nan"), dtype=torch.float32, device=device)
        h.test_activations(dump, k)
    h.run(feats, starts, seeds, N, L, w.gamma, w.lam, out)
    st = h.status()
    if dump is not None:
        h.test_activations(None)
        out["hidden"] = dump
    if st != ROLLOUT_OK:
        raise RolloutError(st, "device-side status")
    if handle is None:
        h.close()
    return out


class PerBuffer:
    """Owns a ``per_buffer`` (include/per.h): the GPU-resident prioritised replay ring."""

    def __init__(self, capacity: int, state_dim: int):
        h = C.c_void_p()
        _check(lib().per_create(int(capacity), int(state_dim), C.byref(h)))
        self._h = h
        self.capacity = int(capacity)
        self.dim = int(state_dim)

    @staticmethod
    def _p(t):
        return C.c_void_p(None) if t is None else C.c_void_p(t.data_ptr())

    def insert(self, states, next_states, actions, rewards, dones, stream=None) -> None:
        """Appends device tensors (states/next_states [n, dim] f32, actions i32,
        rewards f32, dones u8)."""
        p = self._p
        _check(lib().per_insert(self._h, p(states), p(next_states), p(actions), p(rewards), p(dones),
                                int(actions.numel()), C.c_void_p(_stream_handle(stream))))

    def sample(self, batch: int, beta: float, seed: int, offset: int, out: Dict[str, "torch.Tensor"],
               stream=None) -> None:
        """Draws `batch` transitions into the device tensors of `out` (keys indices,
        weights, states, next_states, actions, rewards, dones; the last five optional)."""
        p = self._p
        _check(lib().per_sample(self._h, int(batch), float(beta), C.c_uint64(seed), C.c_uint64(offset),
                                p(out["indices"]), p(out["weights"]), p(out.get("states")),
                                p(out.get("next_states")), p(out.get("actions")), p(out.get("rewards")),
                                p(out.get("dones")), C.c_void_p(_stream_handle(stream))))

    def make_batch(self, batch: int, device="cuda") -> Dict[str, "torch.Tensor"]:
        import torch
        return {"indices": torch.empty(batch, dtype=torch.int32, device=device),
                "weights": torch.empty(batch, dtype=torch.float32, device=device),
                "states": torch.empty((batch, self.dim), dtype=torch.float32, device=device),
                "next_states": torch.empty((batch, self.dim), dtype=torch.float32, device=device),
                "actions": torch.empty(batch, dtype=torch.int32, device=device),
                "rewards": torch.empty(batch, dtype=torch.float32, device=device),
                "dones": torch.empty(batch, dtype=torch.uint8, device=device)}

    def update(self, indices, td_errors, alpha: float = 0.6, eps: float = 1e-6, stream=None) -> None:
        _check(lib().per_update_priorities(self._h, self._p(indices), self._p(td_errors), int(indices.numel()),
                                           float(alpha), float(eps), C.c_void_p(_stream_handle(stream))))

    def size(self):
        n, c = C.c_longlong(), C.c_longlong()
        _check(lib().per_size(self._h, C.byref(n), C.byref(c)))
        return n.value, c.value

    def priorities(self, stream=None):
        """(priorities [capacity] f32, maximum priority) as host values (synchronises)."""
        import numpy as np
        pr = np.empty(self.capacity, dtype=np.float32)
        m = np.empty(1, dtype=np.float32)
        _check(lib().per_read(self._h, pr.ctypes.data_as(C.c_void_p), m.ctypes.data_as(C.c_void_p),
                              C.c_void_p(_stream_handle(stream))))
        return pr, m[0]

    def status(self) -> int:
        return lib().per_status(self._h)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().per_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_dqn_outputs(N: int, L: int, device="cuda", next_states: bool = True) -> Dict[str, "torch.Tensor"]:
    import torch
    f32, i32 = torch.float32, torch.int32
    out = {"states": torch.empty((N, L, wl.STATE_DIM), dtype=f32, device=device),
           "actions": torch.empty((N, L), dtype=i32, device=device),
           "rewards": torch.empty((N, L), dtype=f32, device=device),
           "dones": torch.empty((N, L), dtype=i32, device=device),
           "q": torch.empty((N, L), dtype=f32, device=device),
           "td": torch.empty((N, L), dtype=f32, device=device)}
    if next_states:
        out["next_states"] = torch.empty((N, L, wl.STATE_DIM), dtype=f32, device=device)
    return out


class DqnCollector:
    """Owns a ``dqn_handle`` (include/dqn.h): the DQN experience collector."""

    def __init__(self, weights, dims: RolloutDims):
        import numpy as np
        self._w = np.ascontiguousarray(weights, dtype=np.float32)
        if self._w.size != lib().dqn_weight_count():
            raise ValueError(f"expected {lib().dqn_weight_count()} weights, got {self._w.size}")
        h = C.c_void_p()
        _check(lib().dqn_create(self._w.ctypes.data_as(C.c_void_p), C.byref(dims), C.byref(h)))
        self._h = h

    @classmethod
    def for_workload(cls, w: wl.Workload, weights, n_bars: Optional[int] = None):
        return cls(weights, make_dims(w, n_bars, "bf16"))

    def set_weights(self, weights):
        import numpy as np
        self._w = np.ascontiguousarray(weights, dtype=np.float32)
        _check(lib().dqn_set_weights(self._h, self._w.ctypes.data_as(C.c_void_p)))

    def run(self, features, starts, seeds, N: int, L: int, gamma: float, epsilon: float,
            out: Dict[str, "torch.Tensor"], stream=None) -> None:
        """Enqueues one collection; `out` as make_dqn_outputs (next_states optional)."""
        p = lambda t: C.c_void_p(None) if t is None else C.c_void_p(t.data_ptr())
        _check(lib().dqn_run(self._h, p(features), p(starts), p(seeds), int(N), int(L), float(gamma), float(epsilon),
                             p(out["states"]), p(out["actions"]), p(out["rewards"]), p(out["dones"]), p(out["q"]),
                             p(out["td"]), p(out.get("next_states")), C.c_void_p(_stream_handle(stream))))

    def set_timing(self, on: bool = True) -> None:
        _check(lib().dqn_set_timing(self._h, int(on)))

    def phase_ms(self):
        """Device milliseconds of the last timed run's rollout, state-row and target kernels."""
        ms = (C.c_float * 3)()
        _check(lib().dqn_phase_ms(self._h, ms))
        return [float(x) for x in ms]

    def set_recycle(self, on: bool = True) -> None:
        """Episode recycling: after a done, the next step starts at a fresh bar from the episode's LCG."""
        _check(lib().dqn_set_recycle(self._h, int(on)))

    def test_stall(self, on: bool = True) -> None:
        """Test hook: later runs launch the target pass's stalling test build."""
        _check(lib().dqn_test_stall(self._h, int(on)))

    def status(self) -> int:
        return lib().dqn_status(self._h)

    def close(self):
        if getattr(self, "_h", None) is not None and self._h.value:
            lib().dqn_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
