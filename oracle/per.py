"""Oracle of the GPU-resident prioritised experience replay buffer (include/per.h).

TEST INFRASTRUCTURE ONLY: the tests and the smoke check import this module;
the product path never does.  Plain numpy: double-precision running sums in slot order, one search per
sample, and updates applied as the batch-order writes they define.

Follows page "GPU-Resident Prioritized Experience Replay":
- "New struct: GpuReplayBuffer": the ring's arrays (states, next states,
  actions, rewards, dones, priorities) with the write cursor and the size on
  the host;
- "Experience Insertion": transitions appended at the cursor, which wraps;
  each new transition takes the maximum priority;
- "Sampling Kernels / Proportional": a uniform in [0, total) per sample, the
  cumulative priorities, a search for the slot whose cumulative interval holds
  it, the gather, and the importance-sampling weight
  (1 / (N p_i / total))^beta divided by the largest weight;
- "Priority update": priority = |td|^alpha + epsilon written to the sampled
  slots;
- "Error Handling": non-finite priorities clamped into [epsilon, max priority].
Readings where the page leaves a step open (each stated in the design notes):
the largest weight is taken over the sampled batch; the maximum priority
starts at 1 and is the running maximum of every priority written; within one
update the later entry for a slot wins; a NaN TD error gives epsilon and a
priority past float32 (+inf) the maximum priority held before the update; a
target u total that rounds up to the total is moved just below it; the uniforms come from SplitMix64
(Steele, Lea & Flood, OOPSLA 2014), the (offset + k)-th output for sample k.
"""
from __future__ import annotations

import math
from typing import Optional

import numpy as np

_MASK = (1 << 64) - 1
_GAMMA = 0x9E3779B97F4A7C15


def splitmix64_output(seed: int, n: int) -> int:
    """The n-th output (from 0) of SplitMix64 seeded with `seed`: the state moves
    on by the golden-ratio increment before each output, which is the state run
    through the generator's three xor-shift-multiply mixing steps."""
    z = (seed + (n + 1) * _GAMMA) & _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


def uniform(seed: int, n: int) -> float:
    """The top 53 bits of output n as a double in [0, 1)."""
    return (splitmix64_output(seed, n) >> 11) * 2.0 ** -53


class Replay:
    """The buffer.  state_dim 0 keeps no state rows (for checks of the
    priorities and the sampling alone at large capacities)."""

    def __init__(self, capacity: int, state_dim: int):
        self.capacity = int(capacity)
        self.dim = int(state_dim)
        self.states = np.zeros((capacity, state_dim), dtype=np.float32)
        self.next_states = np.zeros((capacity, state_dim), dtype=np.float32)
        self.actions = np.zeros(capacity, dtype=np.int32)
        self.rewards = np.zeros(capacity, dtype=np.float32)
        self.dones = np.zeros(capacity, dtype=np.uint8)
        self.prio = np.zeros(capacity, dtype=np.float32)
        self.cursor = 0
        self.size = 0
        self.max_prio = np.float32(1.0)
        self.range_error = False

    # -- insertion
    def insert(self, states, next_states, actions, rewards, dones) -> None:
        """Transition j to slot (cursor + j) mod capacity, in order; each takes the
        current maximum priority."""
        count = len(actions)
        # inserted one at a time, only the last `capacity` items survive
        j = np.arange(max(0, count - self.capacity), count)
        s = (self.cursor + j) % self.capacity
        if self.dim:
            self.states[s] = states[j]
            self.next_states[s] = next_states[j]
        self.actions[s] = actions[j]
        self.rewards[s] = rewards[j]
        self.dones[s] = dones[j]
        self.prio[s] = self.max_prio
        self.cursor = (self.cursor + count) % self.capacity
        self.size = min(self.capacity, self.size + count)

    # -- sampling
    def cumulative(self) -> np.ndarray:
        """c_i = p_0 + ... + p_i in double, accumulated in slot order."""
        return np.add.accumulate(self.prio[:self.size].astype(np.float64))

    def sample(self, batch: int, beta: float, seed: int, offset: int, replay: Optional[np.ndarray] = None,
               band: float = 1e-12):
        """Slots, weights and gathered rows of `batch` proportional draws.

        Sample k's slot is the first i with c_i > t_k, t_k = u_k total.  Where t_k
        lies within band * total of a boundary c_i, floating-point summation order
        decides between the two neighbouring slots: if `replay` (another
        implementation's slots) is given, its slot is taken there after checking
        that it is one of the two.  Returns (slots, weights, margins, n_replayed)
        with margins the distance of t_k to the nearest boundary over total."""
        c = self.cumulative()
        total = float(c[-1])
        if not total > 0.0:
            raise ValueError("no positive priority")
        idx = np.zeros(batch, dtype=np.int64)
        margin = np.zeros(batch)
        n_replayed = 0
        for k in range(batch):
            t = uniform(seed, offset + k) * total
            if t >= total:                                     # the product can round up to the total
                t = float(np.nextafter(total, 0.0))
            i = int(np.searchsorted(c, t, side="right"))     # first i with c_i > t
            lo = float(c[i - 1]) if i > 0 else 0.0
            margin[k] = min(t - lo, float(c[i]) - t) / total
            if replay is not None and margin[k] <= band:
                j = int(replay[k])
                assert 0 <= j < self.size and self.prio[j] > 0, (k, j)
                cj_lo = float(c[j - 1]) if j > 0 else 0.0
                assert cj_lo <= t + band * total and float(c[j]) >= t - band * total, (k, i, j)
                if j != i:
                    n_replayed += 1
                i = j
            idx[k] = i
        p = self.prio[idx].astype(np.float64)
        beta = float(np.float32(beta))                         # the ABI takes beta as float32
        w = np.array([(self.size * pk / total) ** (-beta) for pk in p])
        w = (w / w.max()).astype(np.float32)
        return idx, w, margin, n_replayed

    def gather(self, idx):
        return (self.states[idx], self.next_states[idx], self.actions[idx], self.rewards[idx], self.dones[idx])

    # -- priority update
    def update(self, indices, td, alpha: float, eps: float) -> None:
        """p_i = fl32(|td|^alpha + eps) in batch order (the later entry for a slot
        wins); NaN -> eps, +inf -> the maximum priority before the call; the
        maximum priority is the running maximum of the values written."""
        snapshot = self.max_prio
        eps32 = float(np.float32(eps))
        indices = np.asarray(indices, dtype=np.int64)
        ok = (indices >= 0) & (indices < self.size)
        if not ok.all():
            self.range_error = True
        idx = indices[ok]
        d = np.abs(np.asarray(td, dtype=np.float32)[ok].astype(np.float64))
        with np.errstate(over="ignore", invalid="ignore"):     # past float32: +inf, clamped below
            v = (d ** float(np.float32(alpha)) + eps32).astype(np.float32)
        v[np.isnan(d)] = np.float32(eps32)
        v[np.isinf(v)] = snapshot
        # in batch order the last write to a slot stays: keep each slot's last entry
        rev = idx[::-1]
        _, first_in_rev = np.unique(rev, return_index=True)
        last = len(idx) - 1 - first_in_rev
        self.prio[idx[last]] = v[last]
        if len(v):
            self.max_prio = max(self.max_prio, v.max())
