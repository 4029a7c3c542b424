"""Seeded synthetic workloads for fused PPO experience collection.

This module only *generates inputs*: market-feature matrices, episode start
bars, per-episode LCG seeds and initial network weights.  It holds none of the
method's arithmetic (no network, sampler, environment or GAE step), so both the
CUDA path and the CPU oracle can consume the same bytes without sharing code.

Sources for the shapes and distributions ("PPO CUDA Pipeline Design —
Zero-Roundtrip Experience Collection", sections "Kernel Phases" and "Weight
Layout"; the DQN phase-2b page, section "Memory Budget" for the 51 market
features per bar):

* market features ``F[B, 51]`` float32, i.i.d. N(0, 1); column 0 is replaced by
  the bar's log-return ~ N(0, sigma) so that the close price is
  ``P[b] = 100 * exp(cumsum(F[:, 0]))[b]`` and ``P[b+1] / P[b] = exp(F[b+1, 0])``;
* episode starts uniform in ``[0, B - L)`` (overlaps allowed);
* LCG seeds ``seeds[n] = low32(splitmix64(seed * 2**32 + n))`` (SplitMix64 of
  Steele, Lea & Flood 2014 used as the named ``hash(seed, episode)``);
* every weight matrix ``[out, in]`` row-major, He/Kaiming-uniform
  ``U(-sqrt(6/fan_in), +sqrt(6/fan_in))``, every bias zero.

Draw order from ``numpy.random.default_rng(seed)``: features, then column 0,
then starts, then the weights in packing order (actor, critic, curiosity).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Tuple

import numpy as np

N_MARKET = 51          # market features per bar
STATE_DIM = 54         # 51 market + 3 portfolio features
N_ACTIONS = 45         # 5 exposures x 3 order types x 3 urgencies
ACTOR_H = (128, 64)
CRITIC_STD = (512, 384, 256, 128, 64)
CRITIC_WIDE = (1024, 768, 512, 256, 128)
CUR_H = 64             # curiosity forward model: (54 + 45 one-hot) -> 64 -> 54

DTYPES = ("fp32", "tf32", "bf16")


@dataclasses.dataclass(frozen=True)
class Workload:
    """One experience-collection problem: sizes, precision, env constants."""
    name: str
    n_episodes: int            # N
    horizon: int               # L (timesteps per episode)
    n_bars: int                # B (rows of the feature matrix)
    dtype: str                 # "fp32" | "tf32" | "bf16"
    seed: int
    sigma: float               # std of the log-return column
    barrier: float             # +-theta on portfolio PnL since reset
    max_hold: int              # K: time barrier in bars
    gamma: float
    lam: float
    critic_h: Tuple[int, ...] = CRITIC_STD
    # reward / env constants (identical for every workload)
    pt_scale: float = 0.5      # barrier_scale on a profit-take hit
    sl_scale: float = -0.5     # barrier_scale on a stop-loss hit
    div_window: int = 20
    div_thresh: float = 1.0
    div_penalty: float = -0.01
    cur_coef: float = 0.01
    risk_coef: float = 1e-3
    tx_base: float = 1e-4
    spread: float = 1e-4

    @property
    def tuples(self) -> int:
        return self.n_episodes * self.horizon


WORKLOADS: Dict[str, Workload] = {
    # 32 x 200, fp32, 20000 bars, seed 0.
    "tiny_fp32": Workload("tiny_fp32", 32, 200, 20000, "fp32", 0, 1e-3, 0.02, 50, 0.99, 0.95),
    # the pages' default launch: 128 episodes x 500 steps = 64,000 tuples.
    "default_fp32": Workload("default_fp32", 128, 500, 50000, "fp32", 0, 1e-3, 0.02, 50, 0.99, 0.95),
    # 4096 x 500, tf32 tensor-core MLPs, 100000 bars, seed 1.
    "scaleout_tf32": Workload("scaleout_tf32", 4096, 500, 100000, "tf32", 1, 1e-3, 0.02, 50, 0.99, 0.95),
    # 16384 x 1000, bf16, tight barriers (+-0.2 %, 10 bars), sigma 5e-3, seed 2.
    "reset_heavy_bf16": Workload("reset_heavy_bf16", 16384, 1000, 200000, "bf16", 2, 5e-3, 0.002, 10, 0.99, 0.95),
    # 65536 x 256, bf16, widened critic, gamma .995 lambda .97, seed 3.
    "ceiling_bf16": Workload("ceiling_bf16", 65536, 256, 200000, "bf16", 3, 1e-3, 0.02, 50, 0.995, 0.97,
                             critic_h=CRITIC_WIDE),
}
WORKLOAD_ORDER = ["tiny_fp32", "default_fp32", "scaleout_tf32", "reset_heavy_bf16", "ceiling_bf16"]


def layer_shapes(critic_h: Tuple[int, ...] = CRITIC_STD) -> List[Tuple[str, Tuple[int, int]]]:
    """Weight matrices ``(name, (out, in))`` in packing order.

    Packing order is actor W1,b1,W2,b2,W3,b3; critic V1,c1 ... V6,c6; curiosity
    C1,d1,C2,d2.  Each matrix is followed by its bias of length ``out``.
    """
    shapes = [("actor0", (ACTOR_H[0], STATE_DIM)), ("actor1", (ACTOR_H[1], ACTOR_H[0])),
              ("actor2", (N_ACTIONS, ACTOR_H[1]))]
    prev = STATE_DIM
    for i, h in enumerate(critic_h):
        shapes.append((f"critic{i}", (h, prev)))
        prev = h
    shapes.append((f"critic{len(critic_h)}", (1, prev)))
    shapes.append(("cur0", (CUR_H, STATE_DIM + N_ACTIONS)))
    shapes.append(("cur1", (STATE_DIM, CUR_H)))
    return shapes


def n_params(critic_h: Tuple[int, ...] = CRITIC_STD) -> int:
    return sum(o * i + o for _, (o, i) in layer_shapes(critic_h))


def splitmix64(x: int) -> int:
    """SplitMix64 output for state ``x`` (Steele, Lea & Flood, OOPSLA 2014)."""
    m = (1 << 64) - 1
    z = (x + 0x9E3779B97F4A7C15) & m
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & m
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & m
    return z ^ (z >> 31)


def episode_seeds(seed: int, n: int, first: int = 0) -> np.ndarray:
    """``seeds[i] = low32(splitmix64(seed * 2**32 + first + i))`` as uint32 (global
    episode index first + i)."""
    base = (seed & 0xFFFFFFFF) << 32
    return np.array([splitmix64(base + first + i) & 0xFFFFFFFF for i in range(n)], dtype=np.uint32)


def init_weights(rng: np.random.Generator, critic_h: Tuple[int, ...]) -> np.ndarray:
    """Packed float32 buffer of every layer in packing order (He-uniform, zero bias)."""
    parts = []
    for _, (o, i) in layer_shapes(critic_h):
        bound = math.sqrt(6.0 / i)
        parts.append(rng.uniform(-bound, bound, size=(o, i)).astype(np.float32).ravel())
        parts.append(np.zeros(o, dtype=np.float32))
    return np.concatenate(parts)


@dataclasses.dataclass
class Inputs:
    features: np.ndarray       # [B, 51] float32
    starts: np.ndarray         # [N] int32
    seeds: np.ndarray          # [N] uint32
    weights: np.ndarray        # packed float32


def generate(w: Workload, n_episodes: int | None = None, horizon: int | None = None, shard: int = 0) -> Inputs:
    """Seeded synthetic inputs for workload ``w``.

    ``n_episodes``/``horizon`` override N and L (starts are then drawn for the
    overridden sizes); everything else follows the workload's recipe.  ``shard``
    s > 0 gives the s-th block of N episodes of a larger batch (one block per
    process of a multi-GPU run): the same features and weights, the episodes'
    own LCG seeds (global episode indices s*N ..) and start bars (drawn from the
    generator seeded with [seed, s]); shard 0 is the workload's own draw.
    """
    n = w.n_episodes if n_episodes is None else n_episodes
    L = w.horizon if horizon is None else horizon
    rng = np.random.default_rng(w.seed)
    feats = rng.standard_normal((w.n_bars, N_MARKET)).astype(np.float32)
    feats[:, 0] = rng.normal(0.0, w.sigma, size=w.n_bars).astype(np.float32)
    starts = rng.integers(0, w.n_bars - L, size=n).astype(np.int32)
    weights = init_weights(rng, w.critic_h)
    if shard:
        starts = np.random.default_rng([w.seed, shard]).integers(0, w.n_bars - L, size=n).astype(np.int32)
    return Inputs(np.ascontiguousarray(feats), starts, episode_seeds(w.seed, n, first=shard * n), weights)


def weight_views(weights: np.ndarray, critic_h: Tuple[int, ...] = CRITIC_STD) -> Dict[str, np.ndarray]:
    """Named ``[out, in]`` matrix and bias views into a packed buffer."""
    out, off = {}, 0
    for name, (o, i) in layer_shapes(critic_h):
        out[name + ".w"] = weights[off:off + o * i].reshape(o, i)
        off += o * i
        out[name + ".b"] = weights[off:off + o]
        off += o
    assert off == weights.size, (off, weights.size)
    return out


@dataclasses.dataclass(frozen=True)
class ReplayWorkload:
    """A prioritised replay buffer and its training-step traffic."""
    name: str
    capacity: int
    state_dim: int
    batch: int                 # transitions sampled (and priorities updated) per training step
    alpha: float = 0.6
    beta: float = 0.4
    eps: float = 1e-6
    seed: int = 7


REPLAY_WORKLOADS: Dict[str, ReplayWorkload] = {
    # the page's sizing example: 100K transitions
    "replay_100k": ReplayWorkload("replay_100k", 100_000, STATE_DIM, 512),
    # one whole reset-heavy collection (16384 episodes x 1000 steps) held for replay
    "replay_16m": ReplayWorkload("replay_16m", 16_384_000, STATE_DIM, 512),
}


def replay_rows(j: np.ndarray, dim: int):
    """Transition j of the synthetic replay stream, exact in float32 so that a row
    can be recomputed from its index: state[c] = (j mod 65521) + c/64,
    next[c] = (j mod 65519) - c/64, action j mod 45, reward (j mod 1021)/1024,
    done when j mod 7 == 0."""
    j = np.asarray(j, dtype=np.int64)
    c = np.arange(dim, dtype=np.float64) / 64.0
    states = ((j % 65521)[:, None] + c[None, :]).astype(np.float32)
    nxt = ((j % 65519)[:, None] - c[None, :]).astype(np.float32)
    return (states, nxt, (j % 45).astype(np.int32), ((j % 1021) / 1024.0).astype(np.float32),
            (j % 7 == 0).astype(np.uint8))


def replay_td(seed: int, step: int, n: int) -> np.ndarray:
    """Seeded TD errors of one training step: N(0, 1) float32."""
    return np.random.default_rng([seed, step]).standard_normal(n).astype(np.float32)


def replay_rows_device(j0: int, n: int, dim: int, device="cuda"):
    """replay_rows for j = j0 .. j0+n-1, made on the device (same values)."""
    import torch
    j = torch.arange(j0, j0 + n, dtype=torch.int64, device=device)
    c = torch.arange(dim, dtype=torch.float64, device=device) / 64.0
    states = ((j % 65521).to(torch.float64)[:, None] + c[None, :]).to(torch.float32)
    nxt = ((j % 65519).to(torch.float64)[:, None] - c[None, :]).to(torch.float32)
    return (states, nxt, (j % 45).to(torch.int32), ((j % 1021).to(torch.float64) / 1024.0).to(torch.float32),
            (j % 7 == 0).to(torch.uint8))


# ---------------------------------------------------------------- DQN collector

DQN_H, DQN_S = 256, 128     # dueling Q: 54 -> 256 -> 256, then value / advantage streams of 128
DQN_EPSILON = 0.1           # exploration rate of the synthetic launches


def dqn_layer_shapes() -> List[Tuple[str, Tuple[int, int]]]:
    """One dueling Q net's matrices ``(name, (out, in))`` in packing order, each
    followed by its bias: shared W1, W2; value stream Wv1, Wv2; advantage stream
    Wa1, Wa2."""
    return [("q1", (DQN_H, STATE_DIM)), ("q2", (DQN_H, DQN_H)), ("v1", (DQN_S, DQN_H)), ("v2", (1, DQN_S)),
            ("a1", (DQN_S, DQN_H)), ("a2", (N_ACTIONS, DQN_S))]


def dqn_net_params() -> int:
    return sum(o * i + o for _, (o, i) in dqn_layer_shapes())


def dqn_cur_params() -> int:
    return CUR_H * (STATE_DIM + N_ACTIONS) + CUR_H + STATE_DIM * CUR_H + STATE_DIM


# the DQN collector's workloads share the PPO workloads' environments and inputs
DQN_WORKLOADS: Dict[str, Workload] = {
    "dqn_tiny_bf16": dataclasses.replace(WORKLOADS["tiny_fp32"], name="dqn_tiny_bf16", dtype="bf16"),
    "dqn_reset_heavy_bf16": dataclasses.replace(WORKLOADS["reset_heavy_bf16"], name="dqn_reset_heavy_bf16"),
}


def dqn_weights(seed: int, bias_scale: float = 0.0) -> np.ndarray:
    """[online net | target net | curiosity block], float32: He-uniform matrices
    (as init_weights), biases zero or U(-bias_scale, bias_scale).  The target net
    is drawn independently of the online net (not a copy), so that a swap of the
    two shows."""
    rng = np.random.default_rng([seed, 0xD0])
    parts = []
    shapes = dqn_layer_shapes() + dqn_layer_shapes() + [("cur0", (CUR_H, STATE_DIM + N_ACTIONS)),
                                                        ("cur1", (STATE_DIM, CUR_H))]
    for _, (o, i) in shapes:
        bound = math.sqrt(6.0 / i)
        parts.append(rng.uniform(-bound, bound, size=(o, i)).astype(np.float32).ravel())
        b = rng.uniform(-bias_scale, bias_scale, size=o) if bias_scale > 0 else np.zeros(o)
        parts.append(b.astype(np.float32))
    return np.concatenate(parts)
