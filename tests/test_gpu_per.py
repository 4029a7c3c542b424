"""The GPU prioritised replay buffer (include/per.h) against the oracle
(oracle/per.py) on the same seeded transitions and TD errors: ring contents,
sampled slots (exact, except where the target lies within rounding of a
boundary: there the oracle checks the GPU's slot is a neighbour and takes it),
importance weights, gathered rows, priorities and the maximum priority, at
small sizes spanning several blocks with ragged tails and at the benchmark's
full size."""
import numpy as np
import pytest

from rl_experience_collection_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

BAND = 1e-12          # relative to the total: summation-order rounding of doubles
# the weights are formed in float32: x = size p / total (three roundings), log2f
# (1 ulp), the product with beta, exp2f (2 ulp), the division by the batch maximum
# (which carries the same error): below (5 + 1.5 beta |log2 x|) 2^-24 relative,
# 1e-5 for beta |log2 x| up to 60
W_RTOL = 1e-5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from rl_experience_collection_gb300 import build
    build.build()


def _dev(*arrays):
    import torch
    return [torch.from_numpy(np.ascontiguousarray(a)).cuda() for a in arrays]


def _insert(gpu, orc, j0, n, dim):
    rows = wl.replay_rows(np.arange(j0, j0 + n), dim)
    gpu.insert(*_dev(*rows))
    orc.insert(*rows)


def _check_sample(gpu, orc, B, beta, seed, offset):
    out = gpu.make_batch(B)
    gpu.sample(B, beta, seed, offset, out)
    g = {k: v.cpu().numpy() for k, v in out.items()}
    idx, w, margin, n_rep = orc.sample(B, beta, seed, offset, replay=g["indices"], band=BAND)
    far = margin > BAND
    np.testing.assert_array_equal(g["indices"][far], idx[far])
    np.testing.assert_array_equal(g["indices"], idx)        # inside the band the oracle took the GPU's neighbour
    np.testing.assert_allclose(g["weights"], w, rtol=W_RTOL, atol=0)
    s, ns, a, r, d = orc.gather(idx)
    np.testing.assert_array_equal(g["states"], s)
    np.testing.assert_array_equal(g["next_states"], ns)
    np.testing.assert_array_equal(g["actions"], a)
    np.testing.assert_array_equal(g["rewards"], r)
    np.testing.assert_array_equal(g["dones"], d)
    return idx, n_rep


def _check_priorities(gpu, orc):
    pr, m = gpu.priorities()
    assert m == orc.max_prio
    diff = pr.view(np.int32).astype(np.int64) - orc.prio.view(np.int32).astype(np.int64)
    # |td|^alpha + eps is formed in double on both sides and rounded once; the two
    # pow implementations may differ in the last double bit, which can move the
    # float32 rounding by one unit in rare cases
    assert np.abs(diff).max() <= 1
    assert np.count_nonzero(diff) <= max(2, pr.size // 100000)


@pytest.mark.parametrize("C,dim,inserts,B,rounds", [
    (37, 5, [10, 20, 30], 7, 3),                  # tiny ring, two wraps
    (20000, 54, [12000, 12000], 512, 3),          # 3 blocks of 8192, ragged tail, wrapped once
    (5000, 3, [12000], 100, 2),                   # one insert larger than the ring
    (8192 * 3 + 130, 1, [8192 * 3 + 130], 4096, 2),   # full ring, a last block of one sub-block and 2 slots
])
def test_insert_sample_update_match_oracle(C, dim, inserts, B, rounds):
    from rl_experience_collection_gb300 import binding
    from oracle import per
    gpu = binding.PerBuffer(C, dim)
    orc = per.Replay(C, dim)
    j0 = 0
    for n in inserts:
        _insert(gpu, orc, j0, n, dim)
        j0 += n
        assert gpu.size() == (orc.size, orc.cursor)
    _check_priorities(gpu, orc)
    replayed = 0
    for r in range(rounds):
        idx, n_rep = _check_sample(gpu, orc, B, 0.4 + 0.2 * r, seed=11 + r, offset=r * B)
        replayed += n_rep
        td = wl.replay_td(5, r, B)
        idx_dev, td_dev = _dev(idx.astype(np.int32), td)
        gpu.update(idx_dev, td_dev, 0.6, 1e-6)
        orc.update(idx, td, 0.6, 1e-6)
        _check_priorities(gpu, orc)
        _insert(gpu, orc, j0, max(1, C // 7), dim)       # inserts take the running maximum
        j0 += max(1, C // 7)
        _check_priorities(gpu, orc)
    assert replayed <= 2
    assert gpu.status() == binding.ROLLOUT_OK
    gpu.close()


def test_update_edge_cases_and_zero_priorities():
    """Duplicates (the later entry wins), NaN and inf errors, out-of-range slots,
    alpha = 0; zero priorities are never sampled; an all-zero buffer reports."""
    from rl_experience_collection_gb300 import binding
    from oracle import per
    C = 20000
    gpu, orc = binding.PerBuffer(C, 2), per.Replay(C, 2)
    _insert(gpu, orc, 0, C, 2)
    idx = np.array([5, 6, 5, 7, C, -1, 8, 9, 5], dtype=np.int32)
    td = np.array([1.0, np.nan, 4.0, np.inf, 1.0, 1.0, 0.0, 1e30, 9.0], dtype=np.float32)
    for alpha, eps in ((0.6, 0.01), (0.0, 0.5), (2.0, 0.0)):
        gpu.update(*_dev(idx, td), alpha, eps)
        orc.update(idx, td, alpha, eps)
        _check_priorities(gpu, orc)
        assert gpu.status() == binding.ROLLOUT_ERR_RANGE
    # zero out every slot but a scattered few: only those are drawn
    keep = np.array([17, 127, 8191, 8192, 19999])           # sub-block and block edges
    zero = np.setdiff1d(np.arange(C), keep).astype(np.int32)
    for lo in range(0, zero.size, 4000):
        part = zero[lo:lo + 4000]
        gpu.update(*_dev(part, np.zeros(part.size, np.float32)), 1.0, 0.0)
        orc.update(part, np.zeros(part.size, np.float32), 1.0, 0.0)
    _check_priorities(gpu, orc)
    got, _ = _check_sample(gpu, orc, 2000, 0.5, seed=3, offset=0)
    assert set(np.unique(got)) <= set(keep)
    assert gpu.status() == binding.ROLLOUT_OK
    # every priority zero: status word, slot 0, weight 0
    gpu.update(*_dev(keep.astype(np.int32), np.zeros(keep.size, np.float32)), 1.0, 0.0)
    out = gpu.make_batch(16)
    gpu.sample(16, 0.4, 1, 0, out)
    assert gpu.status() == binding.ROLLOUT_ERR_RANGE
    assert (out["indices"].cpu().numpy() == 0).all() and (out["weights"].cpu().numpy() == 0).all()
    gpu.close()


def test_calls_are_deterministic_and_validated():
    import torch
    from rl_experience_collection_gb300 import binding
    res = []
    for _ in range(2):
        gpu = binding.PerBuffer(50000, 4)
        _insert(gpu, __import__("oracle.per", fromlist=["Replay"]).Replay(50000, 4), 0, 50000, 4)
        for r in range(3):
            out = gpu.make_batch(1000)
            gpu.sample(1000, 0.4, 9, r * 1000, out)
            gpu.update(out["indices"], torch.from_numpy(wl.replay_td(1, r, 1000)).cuda())
        pr, m = gpu.priorities()
        res.append((pr, m, out["indices"].cpu().numpy(), out["weights"].cpu().numpy()))
        gpu.close()
    for a, b in zip(res[0], res[1]):
        np.testing.assert_array_equal(a, b)
    with pytest.raises(binding.RolloutError):
        binding.PerBuffer(0, 4)
    gpu = binding.PerBuffer(10, 4)
    out = gpu.make_batch(4)
    with pytest.raises(binding.RolloutError):
        gpu.sample(4, 0.4, 0, 0, out)                      # empty
    _insert(gpu, __import__("oracle.per", fromlist=["Replay"]).Replay(10, 4), 0, 3, 4)
    with pytest.raises(binding.RolloutError):
        gpu.sample(4, -1.0, 0, 0, out)                     # beta < 0
    with pytest.raises(binding.RolloutError):
        gpu.update(out["indices"], out["weights"], alpha=-0.5)
    gpu.close()


def test_full_size_buffer_matches_oracle():
    """The benchmark's buffer (16,384,000 transitions of 54 floats): every slot's
    priority set by 250 updates of 65,536, then batches of 512 compared with the
    oracle (priorities and sampling; the oracle keeps no rows at this size, so the
    gathered rows are checked against the stream's formula for the slot's item)."""
    import torch
    from rl_experience_collection_gb300 import binding
    from oracle import per
    w = wl.REPLAY_WORKLOADS["replay_16m"]
    C, D = w.capacity, w.state_dim
    gpu = binding.PerBuffer(C, D)
    orc = per.Replay(C, 0)
    chunk = 4_096_000
    for j0 in range(0, C, chunk):
        rows = wl.replay_rows_device(j0, chunk, D)
        gpu.insert(*rows)
        orc.insert(None, None, *[r.cpu().numpy() for r in rows[2:]])
        del rows
    torch.cuda.synchronize()
    perm = np.random.default_rng(w.seed).permutation(C).astype(np.int32)
    for k in range(0, C, 65536):
        sl = perm[k:k + 65536]
        td = wl.replay_td(w.seed, 1000 + k // 65536, sl.size)
        gpu.update(*_dev(sl, td), w.alpha, w.eps)
        orc.update(sl, td, w.alpha, w.eps)
    _check_priorities(gpu, orc)
    for r in range(3):
        out = gpu.make_batch(w.batch)
        gpu.sample(w.batch, w.beta, w.seed, r * w.batch, out)
        g = {k: v.cpu().numpy() for k, v in out.items()}
        idx, wt, margin, n_rep = orc.sample(w.batch, w.beta, w.seed, r * w.batch, replay=g["indices"], band=BAND)
        np.testing.assert_array_equal(g["indices"], idx)
        assert n_rep <= 1
        np.testing.assert_allclose(g["weights"], wt, rtol=W_RTOL, atol=0)
        s, ns, a, rw, d = wl.replay_rows(idx, D)                  # slot j holds item j
        np.testing.assert_array_equal(g["states"], s)
        np.testing.assert_array_equal(g["next_states"], ns)
        np.testing.assert_array_equal(g["actions"], a)
        np.testing.assert_array_equal(g["rewards"], rw)
        np.testing.assert_array_equal(g["dones"], d)
        td = wl.replay_td(w.seed, r, w.batch)
        gpu.update(*_dev(idx.astype(np.int32), td), w.alpha, w.eps)
        orc.update(idx, td, w.alpha, w.eps)
    _check_priorities(gpu, orc)
    assert gpu.status() == binding.ROLLOUT_OK
    gpu.close()
