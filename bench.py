"""Benchmark: fused PPO experience collection on GB300.

Default workload: 16384 episodes x 1000 steps, bf16 tensor-core MLPs, 200000
bars x 51 features (the reset-heavy configuration: barriers +-0.2 % / 10 bars,
log-return sigma 5e-3, seed 2).  One step = one rollout_run: rollout
(actor + sample + environment), value (critic + curiosity) and GAE over the
whole batch.  Inputs are resident in HBM; L2 is flushed between timed steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--workload NAME]

Prints one JSON line (rank 0).  --impl reference times the CPU oracle on a
bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import atexit
import dataclasses
import json
import math
import os
import statistics
import subprocess
import tempfile
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from rl_experience_collection_gb300 import workloads as wl  # noqa: E402

METRIC = "experience tuples/sec incl. GAE at 1 GB300; tensor-pipe % of peak"
DEFAULT_WORKLOAD = "reset_heavy_bf16"
ACTOR_FLOP = 2 * (54 * 128 + 128 * 64 + 64 * 45)
CUR_FLOP = 2 * (54 * 64 + 64 * 54)


def critic_flop(h):
    dims = (54,) + tuple(h) + (1,)
    return 2 * sum(a * b for a, b in zip(dims[:-1], dims[1:]))


def path_flops(w: wl.Workload, N: int, L: int):
    """Algorithmic FLOPs of one step (multiply-add = 2): whole path and the value kernel."""
    c = critic_flop(w.critic_h)
    value = N * L * (c + CUR_FLOP) + N * c          # + one bootstrap critic pass per episode
    return N * L * ACTOR_FLOP + value, value


# DRAM bytes (read + write) of one value-kernel launch at the bench's full size,
# scaled from two-counter ncu captures of two small cases of the same workload
# (profiles/ncu_dram_value_umma_reset_heavy_bf16.md: reads fitted as fixed + per
# row, writes at the algorithmic 8 B per row).  A figure only holds for the
# source it was measured on: the sha256 below covers the kernel and the files it
# is built from; any change makes the traffic null.
VALUE_DRAM_CAPTURE = {"workload": "reset_heavy_bf16", "episodes": 16384, "horizon": 1000,
                      "bytes": 526.79e6,
                      "sources_sha256": "5f7775e57cd0bd7d6af9c3467dcc86ba294b2fb5bde442bfc8c2c77a6d79d6fa"}
VALUE_KERNEL_SOURCES = ["value_umma.cu", "umma.cuh", "umma_path.cuh", "env.cuh", "internal.cuh", "umma_pack.cu"]


def value_sources_sha256():
    import hashlib
    hsh = hashlib.sha256()
    csrc = os.path.join(os.path.dirname(os.path.abspath(__file__)), "rl_experience_collection_gb300", "csrc")
    for f in VALUE_KERNEL_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            hsh.update(fh.read())
    return hsh.hexdigest()


PPO_BATCH = 512


def ppo_flop_per_row(critic_h):
    """Multiply-adds of one row through the PPO update's dense products, times 2:
    forward and weight gradient for every layer, input gradient for every layer
    but each network's first."""
    actor = [(54, 128), (128, 64), (64, 45)]
    dims = [54] + list(critic_h) + [1]
    critic = list(zip(dims[:-1], dims[1:]))
    macs = 0
    for net in (actor, critic):
        fwd = sum(i * o for i, o in net)
        macs += 2 * fwd + (fwd - net[0][0] * net[0][1])
    return 2 * macs


def fp32_peak_tflops(sm_mhz):
    """Derived float32 FMA peak: SMs x 128 FP32 lanes x 2 FLOP x clock."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * 128 * 2 * sm_mhz * 1e6 / 1e12


def measure_ppo(w, weights, out, N, L, n_steps, warmup, dev):
    """Times ppo_update on the collected tuples: n_steps Adam steps on mini-batches of
    512 from a seeded permutation, CUDA events on the launching stream."""
    import torch
    from rl_experience_collection_gb300 import binding
    T = N * L
    tr = binding.PpoTrainer.for_workload(w, weights)
    states = out["states"].reshape(-1, 54)
    actions, logp, adv, ret = (out[k].reshape(-1) for k in ("actions", "logp", "adv", "ret"))
    rng = np.random.default_rng(5)
    idx = torch.from_numpy(rng.choice(T, size=(warmup + n_steps) * PPO_BATCH, replace=False).astype(np.int32)).to(dev)
    stream = torch.cuda.current_stream(dev)
    timed = idx[warmup * PPO_BATCH:]
    # the warm-up call uses the timed call's arrays, so that the step graph it
    # captures is the one the timed call replays
    tr.update(states, actions, logp, adv, ret, timed, warmup, PPO_BATCH, stream=stream)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    tr.update(states, actions, logp, adv, ret, timed, n_steps, PPO_BATCH, stream=stream)
    e1.record(stream)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / n_steps
    if tr.status() != binding.ROLLOUT_OK:
        raise SystemExit("PPO update status")
    tr.close()
    flop = ppo_flop_per_row(w.critic_h) * PPO_BATCH
    return ms, flop


REPLAY_BATCH = 512


def measure_replay(out, N, L, dev, flush, iters):
    """The prioritised replay buffer holding this collection (capacity N x L):
    one insert of every tuple (next state = the episode's following row; the
    last row repeats), priorities set from the advantages, then `iters` training
    steps of one 512-sample draw and one 512-entry priority update, each call
    timed with CUDA events after an L2 flush."""
    import torch
    from rl_experience_collection_gb300 import binding
    T, D = N * L, wl.STATE_DIM
    stream = torch.cuda.current_stream(dev)
    states = out["states"].reshape(N, L, D)
    nxt = torch.cat([states[:, 1:], states[:, -1:]], dim=1).reshape(T, D)
    states = states.reshape(T, D)
    actions, rewards = out["actions"].reshape(-1), out["rewards"].reshape(-1)
    dones = out["dones"].reshape(-1).to(torch.uint8)
    buf = binding.PerBuffer(T, D)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ins = []
    for i in range(3):
        flush.fill_(float(i))
        e0.record(stream)
        buf.insert(states, nxt, actions, rewards, dones, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        ins.append(e0.elapsed_time(e1))
    del nxt
    adv = out["adv"].reshape(-1)
    perm = torch.from_numpy(np.random.default_rng(3).permutation(T).astype(np.int32)).to(dev)
    for k in range(0, T, 65536):
        sl = perm[k:k + 65536]
        buf.update(sl, adv[sl.long()], stream=stream)
    batch = buf.make_batch(REPLAY_BATCH, dev)
    td = torch.randn((iters + 3, REPLAY_BATCH), generator=torch.Generator(device=dev).manual_seed(9), device=dev)
    samp, upd = [], []
    for i in range(iters + 3):
        flush.fill_(float(i))
        e0.record(stream)
        buf.sample(REPLAY_BATCH, 0.4, 17, i * REPLAY_BATCH, batch, stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        t_s = e0.elapsed_time(e1)
        flush.fill_(float(i))
        e0.record(stream)
        buf.update(batch["indices"], td[i], stream=stream)
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 3:
            samp.append(t_s)
            upd.append(e0.elapsed_time(e1))
    if buf.status() != binding.ROLLOUT_OK:
        raise SystemExit("replay status")
    buf.close()
    return statistics.median(ins), statistics.median(samp), statistics.median(upd)


def replay_insert_bytes(T, D):
    """Algorithmic bytes of inserting T transitions: rows, action, reward, done
    read and written, the priority written, the new priorities read once by the
    sub-block sums."""
    row = 2 * D * 4 + 4 + 4 + 1
    return 2 * T * row + T * 4 + T * 4


def replay_sample_bytes(B, D, n_blocks):
    """Algorithmic bytes of one sampling call: per sample the 32-way search over
    the block prefix (32 doubles a round), 16 sub-sums, 128 priorities, the
    gathered transition read and written, the slot and weight written (and the
    weight read and rewritten by the normalisation)."""
    rounds = max(1, math.ceil(math.log(max(n_blocks, 2), 32)))
    row = 2 * D * 4 + 4 + 4 + 1
    return B * (rounds * 32 * 8 + 16 * 8 + 128 * 4 + 2 * row + 4 + 8 + 8 + 4)


DQN_NET_FLOP = 2 * (54 * 256 + 256 * 256 + 2 * 256 * 128 + 128 + 45 * 128)   # one dueling Q pass, valid dims
DQN_CUR_FLOP = 2 * (54 * 64 + 64 * 54)                                    # curiosity (one-hot column adds not counted)


def measure_dqn(dev, flush, steps, warmup):
    """The DQN collector on the reset-heavy environment at full size (16384 x 1000,
    bf16): CUDA events around each run (L2 flushed before it) and per-kernel times,
    without and with episode recycling: {False: (ms, phases), True: (ms, phases)}."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.DQN_WORKLOADS["dqn_reset_heavy_bf16"]
    N, L = w.n_episodes, w.horizon
    inp = wl.generate(w)
    h = binding.DqnCollector.for_workload(w, wl.dqn_weights(w.seed, 0.05))
    out = binding.make_dqn_outputs(N, L, dev, next_states=False)
    stream = torch.cuda.current_stream(dev)
    args = (torch.from_numpy(inp.features).to(dev), torch.from_numpy(inp.starts).to(dev),
            torch.from_numpy(inp.seeds.view(np.int32)).to(dev), N, L, w.gamma, wl.DQN_EPSILON, out, stream)
    res = {}
    for recycle in (False, True):
        h.set_recycle(recycle)
        h.set_timing(False)
        for _ in range(warmup):
            h.run(*args)
        torch.cuda.synchronize()
        h.set_timing(True)
        ms, phase = [], []
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        for i in range(steps):
            flush.fill_(float(i))
            e0.record(stream)
            h.run(*args)
            e1.record(stream)
            phase.append(h.phase_ms())
            ms.append(e0.elapsed_time(e1))
        if h.status() != binding.ROLLOUT_OK:
            raise SystemExit("DQN status")
        res[recycle] = (statistics.mean(ms), [statistics.mean(p[i] for p in phase) for i in range(3)])
    h.close()
    return w, res


OTHER_WORKLOADS = ("scaleout_tf32", "ceiling_bf16")


def measure_workload(name: str, dev, flush, steps: int, warmup: int):
    """One more workload timed like the main line (inputs resident, warm-up,
    L2 flushed before every step, CUDA events on the launching stream) with its
    value kernel's roofline against the tensor peak of its operand type."""
    import torch
    from rl_experience_collection_gb300 import binding
    w = wl.WORKLOADS[name]
    N, L = w.n_episodes, w.horizon
    inputs = wl.generate(w)
    h = binding.Rollout.for_workload(w, inputs.weights)
    feats = torch.from_numpy(inputs.features).to(dev)
    starts = torch.from_numpy(inputs.starts).to(dev)
    seeds = torch.from_numpy(inputs.seeds.view(np.int32)).to(dev)
    out = binding.make_outputs(N, L, dev)
    stream = torch.cuda.current_stream(dev)
    for _ in range(warmup):
        h.run(feats, starts, seeds, N, L, w.gamma, w.lam, out, stream)
    torch.cuda.synchronize()
    h.set_timing(True)
    ms, phase = [], []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(steps):
        flush.fill_(float(i))
        e0.record(stream)
        h.run(feats, starts, seeds, N, L, w.gamma, w.lam, out, stream)
        e1.record(stream)
        phase.append(h.phase_ms())
        ms.append(e0.elapsed_time(e1))
    if h.status() != binding.ROLLOUT_OK:
        raise SystemExit(f"{name}: device status")
    h.close()
    del out
    torch.cuda.empty_cache()
    pk = peaks()
    tpk, tpk_name = tensor_peak(w.dtype, pk)
    flop_step, flop_value = path_flops(w, N, L)
    step_ms = statistics.mean(ms)
    pm = {k: statistics.mean(p[i] for p in phase) for i, k in enumerate(("rollout", "states", "value", "gae"))}
    achieved = flop_value / (pm["value"] / 1000.0) / 1e12
    return {"workload": f"{name}: {N} x {L}, {w.dtype}, critic {'/'.join(map(str, w.critic_h))}",
            "tuples_per_s": N * L / (step_ms / 1000.0), "ms_per_step": step_ms, "steps": steps, "warmup": warmup,
            "phase_ms": pm,
            "roofline": {"kernel": "value (critic + curiosity, tcgen05; activations in per-CTA L2 scratch)",
                         "bound": "tensor", "achieved": achieved, "peak": tpk, "unit": "TFLOP/s",
                         "frac": achieved / tpk, "peak_kind": f"{tpk_name}, burst, {pk['src']}",
                         "algorithmic_flop_per_launch": flop_value, "traffic": None},
            "tensor_pipe_frac_step": flop_step / (step_ms / 1000.0) / 1e12 / tpk,
            "gpu_launches": launches_per_run(w.dtype) * steps, "l2": "flushed between steps"}


def launches_per_run(dtype):
    """Kernels one rollout_run launches: feature padding (bf16 only), rollout,
    state rows, value, GAE."""
    return 5 if dtype == "bf16" else 4


def value_dram_traffic(w, N, L):
    c = VALUE_DRAM_CAPTURE
    if c["bytes"] is None or (w.name, N, L) != (c["workload"], c["episodes"], c["horizon"]):
        return None
    return c["bytes"] if value_sources_sha256() == c["sources_sha256"] else None


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return {"bf16": d["bf16_tflops"], "bf16_sustained": d.get("bf16_tflops_sustained"),
                "hbm": d["hbm_gbs"], "src": "measured"}
    return {"bf16": 1900.0, "bf16_sustained": 1700.0, "hbm": 6800.0, "src": "fallback"}


def tensor_peak(dtype: str, pk):
    # tf32 dense rate is half of bf16's (nominal ratio); fp32 runs on CUDA cores
    if dtype == "bf16":
        return pk["bf16"], "bf16"
    if dtype == "tf32":
        return pk["bf16"] / 2.0, "tf32 (= measured bf16 x nominal 1/2)"
    return None, "fp32 CUDA cores"


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 50 ms.

    Started before the warm-up, so that nvidia-smi is already sampling when the
    timed region begins; mark() brackets that region with the host's wall clock,
    and summary() keeps the samples whose nvidia-smi timestamps fall inside it
    (or, where a timestamp does not parse, the lines written after the region
    began)."""
    Q = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")
    TS_FORMAT = "%Y/%m/%d %H:%M:%S.%f"

    def __init__(self, index: int, interval_ms: int = 50, exe: str = "nvidia-smi"):
        self.index, self.interval_ms, self.exe = index, interval_ms, exe
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"bench_clocks_{os.getpid()}.csv")   # transient
        self.t0 = self.t1 = None
        self.lines_at_t0 = 0

    def start(self, settle_s: float = 2.0):
        """Starts sampling and waits (at most settle_s) for the first sample."""
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen([self.exe, f"--id={self.index}", f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.interval_ms)],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            return self
        end = time.time() + settle_s
        while time.time() < end and self.proc.poll() is None and os.path.getsize(self.path) == 0:
            time.sleep(0.01)
        return self

    def _lines(self):
        try:
            return open(self.path).read().strip().splitlines()
        except OSError:
            return []

    def mark(self, begin: bool):
        """Brackets the timed region (call with True just before it, False just after)."""
        if begin:
            self.t0 = time.time()
            self.lines_at_t0 = len(self._lines())
        else:
            self.t1 = time.time()
            time.sleep(2.5 * self.interval_ms / 1000.0)    # the sample taken at the region's end

    def stop(self):
        if not self.proc:
            return
        if self.proc.poll() is None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=10)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
        if not self.f.closed:
            self.f.close()

    def _in_region(self, rows):
        import datetime
        slack = self.interval_ms / 1000.0
        try:
            ts = [datetime.datetime.strptime(r[0].strip(), self.TS_FORMAT).timestamp() for r in rows]
        except ValueError:
            return rows[self.lines_at_t0:], "lines written after the region began"
        if self.t0 is None or self.t1 is None:
            return rows, "whole run"
        sel = [r for r, t in zip(rows, ts) if self.t0 - slack <= t <= self.t1 + slack]
        return sel, "timed region"

    def summary(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]}
        rows = [r.split(",") for r in self._lines() if r.count(",") >= 8]
        try:
            os.remove(self.path)
        except OSError:
            pass
        rows, window = self._in_region(rows)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "window": window}
        try:
            sm = [float(r[1]) for r in rows]
            names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
            reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
            return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]), "reasons": reasons,
                    "samples": len(rows), "window": window, "interval_ms": self.interval_ms,
                    "power_w_median": statistics.median(float(r[3]) for r in rows),
                    "power_w_max": max(float(r[3]) for r in rows)}
        except (ValueError, IndexError):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unparsed samples"], "window": window}


def profile_run(kind: str, episodes: int, horizon: int) -> None:
    """A fixed sequence of library calls for an ``ncu`` capture (no timing, no
    JSON line): ``dqn`` creates the DQN collector for the reset-heavy workload
    and runs it three times on ``episodes`` x ``horizon``; ``replay`` fills a
    16,384,000-slot buffer of one-float states, gives every slot a priority in
    250 updates of 65,536, then makes five draws of 512 each followed by its
    priority update.  Ends with the handle's status check."""
    import torch
    from rl_experience_collection_gb300 import binding, build
    build.build()
    if kind == "dqn":
        w = wl.DQN_WORKLOADS["dqn_reset_heavy_bf16"]
        N, L = episodes or 2048, horizon or 200
        inp = wl.generate(w, n_episodes=N, horizon=L)
        h = binding.DqnCollector.for_workload(w, wl.dqn_weights(w.seed, 0.05))
        out = binding.make_dqn_outputs(N, L, next_states=False)
        args = (torch.from_numpy(inp.features).cuda(), torch.from_numpy(inp.starts).cuda(),
                torch.from_numpy(inp.seeds.view(np.int32)).cuda(), N, L, w.gamma, wl.DQN_EPSILON, out)
        for _ in range(3):
            h.run(*args)
        torch.cuda.synchronize()
        st = h.status()
    else:
        C, D, U = 16_384_000, 1, 65_536
        buf = binding.PerBuffer(C, D)
        buf.insert(*wl.replay_rows_device(0, C, D))
        g = torch.Generator(device="cuda").manual_seed(1)
        perm = torch.randperm(C, device="cuda", generator=g).int()
        for k in range(0, C, U):
            buf.update(perm[k:k + U], torch.randn(U, device="cuda", generator=g))
        batch = buf.make_batch(512)
        for i in range(5):
            buf.sample(512, 0.4, 17, i * 512, batch)
            buf.update(batch["indices"], torch.randn(512, device="cuda", generator=g))
        torch.cuda.synchronize()
        st = buf.status()
    if st != binding.ROLLOUT_OK:
        raise SystemExit(f"device status {st}")
    print("ok")


def dist_setup(backend: str = "nccl"):
    """(rank, world size, torch.distributed or None) from the launcher's environment
    (RANK, WORLD_SIZE, MASTER_ADDR, MASTER_PORT); one process per GPU."""
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, None
    import torch.distributed as dist
    dist.init_process_group(backend)
    return dist.get_rank(), ws, dist


def max_over_ranks(x: float, dist, device):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def host_cpu():
    """The host's logical CPU count and CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except OSError:
            pass
    import platform
    return {"nproc": os.cpu_count(), "model": model or platform.machine()}


def run_oracle_sample(w: wl.Workload, inputs, n_eps: int, first: int = 0, threads: int = 1):
    """Times the oracle (as it stands) on episodes first .. first+n_eps-1, episode-
    parallel over `threads` host threads (the C calls release the GIL)."""
    from oracle import oracle as orc
    idx = [(first + i) % w.n_episodes for i in range(n_eps)]
    t0 = time.perf_counter()
    orc.rollout(w, inputs, idx, quant=w.dtype, threads=threads)
    return time.perf_counter() - t0, n_eps * w.horizon


def workload_config(w: wl.Workload, n_episodes: int, horizon: int, world: int) -> dict:
    """The `config` object of both arms' JSON lines (the same dict for the same
    workload, so the two lines compare)."""
    return {"workload": w.name, "episodes": n_episodes, "horizon": horizon, "n_bars": w.n_bars,
            "critic": list(w.critic_h), "l2": "flushed between steps (512 MB write)",
            "parallelism": "replicas" if world > 1 else "single GPU"}


def reference_arm(args, w: wl.Workload, rank: int):
    if rank != 0:
        return
    inputs = wl.generate(w)
    cpu = host_cpu()
    threads = max(1, cpu["nproc"] or 1)
    n_eps = max(1, int(args.ref_episodes)) * threads
    for i in range(args.warmup):
        run_oracle_sample(w, inputs, n_eps, first=i * n_eps, threads=threads)
    times, tuples = [], 0
    for i in range(args.steps):
        dt, n = run_oracle_sample(w, inputs, n_eps, first=(args.warmup + i) * n_eps, threads=threads)
        times.append(dt)
        tuples += n
    v = tuples / sum(times)
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tuples/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * sum(times) / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": workload_config(w, w.n_episodes, w.horizon, args.gpus),
            "cpu_baseline": {"value": v, "unit": "tuples/s", "cores": threads, "kind": "oracle",
                             "nproc": cpu["nproc"], "cpu_model": cpu["model"],
                             "sample": f"{n_eps} episodes x {w.horizon} steps per step, episode-parallel "
                                       f"over {threads} threads"},
            "e2e": {"value": v, "unit": "tuples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(wl.WORKLOADS))
    ap.add_argument("--ref-episodes", type=int, default=1, help="oracle episodes per host thread per reference step")
    ap.add_argument("--cpu-episodes", type=int, default=256, help="oracle episodes for cpu_baseline (all host cores)")
    ap.add_argument("--no-others", action="store_true",
                    help="skip the measurements of the tf32 and widened-critic workloads")
    ap.add_argument("--episodes", type=int, default=None,
                    help="override the workload's episode count (a smaller case for profiling)")
    ap.add_argument("--horizon", type=int, default=None, help="override the workload's horizon")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-ppo", action="store_true", help="skip the PPO-update measurement")
    ap.add_argument("--ppo-steps", type=int, default=200, help="timed PPO optimizer steps (mini-batches of 512)")
    ap.add_argument("--no-replay", action="store_true", help="skip the prioritised-replay measurement")
    ap.add_argument("--replay-steps", type=int, default=200, help="timed replay sample + update calls")
    ap.add_argument("--no-dqn", action="store_true", help="skip the DQN-collector measurement")
    ap.add_argument("--profile", choices=["dqn", "replay"],
                    help="run a fixed call sequence for an ncu capture instead of the benchmark")
    args = ap.parse_args()
    if args.profile:
        profile_run(args.profile, args.episodes, args.horizon)
        return
    args.warmup = max(args.warmup, 3)
    w = wl.WORKLOADS[args.workload]
    if args.episodes or args.horizon:
        w = dataclasses.replace(w, n_episodes=args.episodes or w.n_episodes, horizon=args.horizon or w.horizon)

    # the reference arm is host work on every rank: gloo, so that no rank touches a GPU
    rank, world, dist = dist_setup("gloo" if args.impl == "reference" else "nccl")
    if args.impl == "reference":
        reference_arm(args, w, rank)
        if dist is not None:
            dist.barrier()
        return

    import torch
    from rl_experience_collection_gb300 import binding, build
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if rank == 0 or world == 1:
        build.build()
    if dist is not None:
        dist.barrier()
    N, L = w.n_episodes, w.horizon
    inputs = wl.generate(w, shard=rank)          # this rank's episodes (weak scaling: N per GPU)
    h = binding.Rollout.for_workload(w, inputs.weights)
    feats = torch.from_numpy(inputs.features).to(dev)
    starts = torch.from_numpy(inputs.starts).to(dev)
    seeds = torch.from_numpy(inputs.seeds.view(np.int32)).to(dev)
    out = binding.make_outputs(N, L, dev)
    flush = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)   # 512 MB > L2
    stream = torch.cuda.current_stream(dev)

    def step():
        h.run(feats, starts, seeds, N, L, w.gamma, w.lam, out, stream)

    clk = ClockSampler(torch.cuda.current_device()).start()
    atexit.register(clk.stop)                    # no sampler outlives the run
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    st = h.status()
    if st != binding.ROLLOUT_OK:
        clk.stop()
        raise SystemExit(f"device status {st} after warm-up")

    # ---------------- device-resident timing (per step, L2 flushed between steps)
    h.set_timing(True)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    phase = []
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    clk.mark(True)
    try:
        for i in range(args.steps):
            flush.fill_(float(i))
            ev[i][0].record(stream)
            step()
            ev[i][1].record(stream)
            phase.append(h.phase_ms())
        torch.cuda.synchronize()
        clk.mark(False)
    finally:
        clk.stop()
    if dist is not None:
        dist.barrier()
    h.set_timing(False)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    total_ms = max_over_ranks(sum(step_ms), dist, dev)
    st = h.status()
    if st != binding.ROLLOUT_OK:
        raise SystemExit(f"device status {st} after the timed steps")
    ms = total_ms / args.steps
    tuples = N * L * world
    value = tuples * args.steps / (total_ms / 1000.0)

    pk = peaks()
    flop_step, flop_value = path_flops(w, N, L)
    tpk, tpk_name = tensor_peak(w.dtype, pk)
    rollout_ms = statistics.mean(p[0] for p in phase)
    states_ms = statistics.mean(p[1] for p in phase)
    value_ms = statistics.mean(p[2] for p in phase)
    gae_ms = statistics.mean(p[3] for p in phase)
    achieved = flop_value / (value_ms / 1000.0) / 1e12
    roofline = {"kernel": "value (critic + curiosity, tcgen05)", "bound": "tensor", "achieved": achieved,
                "peak": tpk, "unit": "TFLOP/s", "frac": (achieved / tpk) if tpk else None,
                "traffic": value_dram_traffic(w, N, L),
                "peak_kind": f"{tpk_name}, burst, {pk['src']}",
                "algorithmic_flop_per_launch": flop_value}
    line = {"metric": METRIC, "value": value, "unit": "tuples/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": w.dtype, "data": "synthetic",
            "config": workload_config(w, N, L, world),
            "tensor_pipe_frac_step": (flop_step / (ms / 1000.0) / 1e12 / tpk) if tpk else None,
            "phase_ms": {"rollout": rollout_ms, "states": states_ms, "value": value_ms, "gae": gae_ms},
            "roofline": roofline, "clocks": clk.summary(), "gpu_launches": launches_per_run(w.dtype) * args.steps}

    # ---------------- the tf32 and widened-critic workloads (rank 0 alone)
    if not args.no_others and rank == 0 and args.workload == DEFAULT_WORKLOAD and not (args.episodes or args.horizon):
        line["workloads"] = {}
        for name in OTHER_WORKLOADS:
            line["workloads"][name] = measure_workload(name, dev, flush, args.steps, args.warmup)

    # ---------------- the PPO update on the collected tuples (rank 0 alone, float32)
    if not args.no_ppo and rank == 0:
        ms, flop = measure_ppo(w, inputs.weights, out, N, L, args.ppo_steps, 10, dev)
        peak = fp32_peak_tflops(line["clocks"].get("sm_max_mhz") or 2070.0)
        achieved = flop / (ms / 1000.0) / 1e12
        line["ppo_update"] = {"batch": PPO_BATCH, "steps": args.ppo_steps, "ms_per_step": ms,
                              "tuples_per_s": PPO_BATCH / (ms / 1000.0), "flop_per_step": flop,
                              "achieved_tflops": achieved, "peak_tflops": peak,
                              "peak_kind": "fp32 FMA, derived: SMs x 128 lanes x 2 x max SM clock",
                              "frac": achieved / peak, "bound": "alu"}

    # ---------------- the prioritised replay buffer holding this collection (rank 0)
    if not args.no_replay and rank == 0:
        ins_ms, s_ms, u_ms = measure_replay(out, N, L, dev, flush, args.replay_steps)
        T, D = N * L, wl.STATE_DIM
        ib = replay_insert_bytes(T, D)
        sb = replay_sample_bytes(REPLAY_BATCH, D, (T + 2047) // 2048)
        line["replay"] = {
            "workload": f"capacity {T} (this collection), state_dim {D}, batch {REPLAY_BATCH}, alpha 0.6, beta 0.4",
            "insert_ms": ins_ms, "sample_us": 1000 * s_ms, "update_us": 1000 * u_ms,
            "samples_per_s": REPLAY_BATCH / (s_ms / 1000.0),
            "insert_roofline": {"bound": "hbm", "achieved": ib / (ins_ms / 1000.0) / 1e9, "peak": pk["hbm"],
                                "unit": "GB/s", "frac": ib / (ins_ms / 1000.0) / 1e9 / pk["hbm"],
                                "algorithmic_bytes": ib},
            "sample_roofline": {"bound": "latency", "achieved": sb / (s_ms / 1000.0) / 1e9, "peak": pk["hbm"],
                                "unit": "GB/s", "frac": sb / (s_ms / 1000.0) / 1e9 / pk["hbm"],
                                "algorithmic_bytes": sb},
            "gpu_launches_per_step": 7, "l2": "flushed before every timed call"}

    # ---------------- the DQN collector on the same environment (rank 0)
    if not args.no_dqn and rank == 0:
        del out
        out = None
        torch.cuda.empty_cache()
        dw, dres = measure_dqn(dev, flush, args.steps, args.warmup)
        d_ms, (r_ms, s_ms, t_ms) = dres[False]
        dr_ms, dr_phase = dres[True]
        T = dw.n_episodes * dw.horizon
        r_fl, t_fl = T * DQN_NET_FLOP, T * (DQN_NET_FLOP + DQN_CUR_FLOP)
        peak_b = pk["bf16"]
        line["dqn"] = {
            "workload": f"{dw.name}: {dw.n_episodes} x {dw.horizon}, epsilon {wl.DQN_EPSILON}, bf16",
            "tuples_per_s": T / (d_ms / 1000.0), "ms_per_run": d_ms,
            "phase_ms": {"rollout": r_ms, "states": s_ms, "target": t_ms},
            "rollout_roofline": {"bound": "tensor", "achieved": r_fl / (r_ms / 1000.0) / 1e12, "peak": peak_b,
                                 "unit": "TFLOP/s", "frac": r_fl / (r_ms / 1000.0) / 1e12 / peak_b,
                                 "algorithmic_flop_per_launch": r_fl},
            "target_roofline": {"bound": "tensor", "achieved": t_fl / (t_ms / 1000.0) / 1e12, "peak": peak_b,
                                "unit": "TFLOP/s", "frac": t_fl / (t_ms / 1000.0) / 1e12 / peak_b,
                                "algorithmic_flop_per_launch": t_fl},
            "gpu_launches_per_run": 4, "l2": "flushed between runs",
            "recycle": {"tuples_per_s": T / (dr_ms / 1000.0), "ms_per_run": dr_ms,
                        "phase_ms": dict(zip(("rollout", "states", "target"), dr_phase))}}
        out = binding.make_outputs(N, L, dev)

    # ---------------- end to end through the C ABI with host buffers (rollout_run_host:
    # inputs copied in, every output copied back as soon as its kernel is done)
    if not args.no_e2e:
        h.set_timing(False)
        hf = torch.from_numpy(inputs.features).pin_memory()
        hs = torch.from_numpy(inputs.starts).pin_memory()
        hd = torch.from_numpy(inputs.seeds.view(np.int32)).pin_memory()
        keep = ("states", "actions", "logp", "adv", "ret", "dones", "rewards")
        hout = {k: torch.empty(out[k].shape, dtype=out[k].dtype, pin_memory=True) for k in keep}
        h2d = hf.numel() * 4 + hs.numel() * 4 + hd.numel() * 4
        d2h = sum(t.numel() * 4 for t in hout.values())
        e2e_ms = []
        for i in range(args.warmup + args.steps):
            flush.fill_(float(i))
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            h.run_host(hf, hs, hd, N, L, w.gamma, w.lam, hout, stream)
            torch.cuda.synchronize()
            if i >= args.warmup:
                e2e_ms.append(1000 * (time.perf_counter() - t0))
        if h.status() != binding.ROLLOUT_OK:
            raise SystemExit("device status after the end-to-end runs")
        e2e_total = max_over_ranks(sum(e2e_ms), dist, dev)
        line["e2e"] = {"value": tuples * args.steps / (e2e_total / 1000.0), "unit": "tuples/s",
                       "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # ---------------- CPU oracle baseline (rank 0, N=1 only)
    if rank == 0 and world == 1 and not args.no_cpu:
        cpu = host_cpu()
        threads = max(1, cpu["nproc"] or 1)
        dt, n = run_oracle_sample(w, inputs, args.cpu_episodes, threads=threads)
        dt1, n1 = run_oracle_sample(w, inputs, 4, first=args.cpu_episodes)
        line["cpu_baseline"] = {"value": n / dt, "unit": "tuples/s", "cores": threads, "kind": "oracle",
                                "nproc": cpu["nproc"], "cpu_model": cpu["model"],
                                "single_thread_value": n1 / dt1,
                                "sample": f"first {args.cpu_episodes} episodes x {L} steps of {w.name}, "
                                          f"{w.dtype} operand rounding, episode-parallel over {threads} "
                                          f"threads, {dt:.1f} s (single thread: 4 episodes, {dt1:.1f} s)"}
    h.close()
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
