/*
 * dqn.h -- C ABI of the DQN experience collector: N independent episodes step
 * through L timesteps of the same environment as the PPO collector
 * (rollout.h), choosing each action epsilon-greedily from a dueling Q
 * network, and every transition gets its TD error from a target network, for
 * prioritised replay (per.h).  No host round trip inside a run.
 *
 * Defining passage: page "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA
 * Experience Collection", "Data Flow" (per step: features, portfolio
 * features, online Q forward, epsilon-greedy selection with the LCG,
 * portfolio, barrier, diversity, curiosity, next state, target Q forward, TD
 * error, reward, store, reset on done) and "Kernel Components" 1 (dueling Q:
 * 54 -> 256 LeakyReLU(0.01) -> 256 LeakyReLU(0.01); value stream 256 -> 128
 * LeakyReLU -> 1; advantage stream 256 -> 128 LeakyReLU -> 45;
 * Q = V + (A - mean A)), 7 (TD error) and 8 (LCG).
 *
 * Per step, with u1, u2 the next two LCG uniforms of the episode (the
 * generator of rollout.h, s = s * 1664525 + 1013904223, u = (s >> 8) 2^-24):
 *   a = u1 < epsilon ? floor(u2 * 45) : the first index of max_a Q_online(x, a)
 *   environment step, curiosity bonus and reward exactly as rollout.h;
 *   q  = Q_online(x, a);  x' = the pre-reset next state [F[b+1], V', e', spread]
 *   td = | r + gamma * max_a Q_target(x', a) * (1 - done) - q |.
 * Both networks run on tcgen05 tensor cores with bf16 operands (weights and
 * each layer's input rounded to bf16, round to nearest even) and float32
 * accumulation; biases, activations, the dueling combination and the
 * environment are float32.
 *
 * Weights (host, float32, dqn_weight_count() floats): [online net | target net
 * | curiosity block]; each net W1 [256 x 54], b1, W2 [256 x 256], b2,
 * Wv1 [128 x 256], bv1, Wv2 [1 x 128], bv2, Wa1 [128 x 256], ba1,
 * Wa2 [45 x 128], ba2 (row-major [out, in], each matrix followed by its
 * bias); the curiosity block C1 [64 x 99], c1, C2 [54 x 64], c2 as in the PPO
 * layout.
 *
 * Thread-compatible, not thread-safe: calls on one handle must be ordered.
 */
#ifndef DQN_H
#define DQN_H

#include <stdint.h>

#include "rollout.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct dqn_handle dqn_handle;

/* floats in the packed weight buffer (2 x 151,598 + 9,910) */
ROLLOUT_API long long dqn_weight_count(void);

/*
 * dqn_create -- converts the weights (host, copied) for the tensor cores.
 * dims: n_market 51, n_actions 45, cur_h 64, dtype ROLLOUT_BF16, n_bars and
 * the environment constants as rollout_create takes them (the actor and
 * critic fields are ignored).  Returns ROLLOUT_OK, _INVALID, _UNSUPPORTED,
 * _NOMEM or _CUDA.
 */
ROLLOUT_API int dqn_create(const float *weights, const rollout_dims *dims, dqn_handle **out);

/* dqn_set_weights -- replaces online, target and curiosity weights (host
 * buffer, copied); synchronous.  Returns ROLLOUT_OK, _INVALID or _CUDA. */
ROLLOUT_API int dqn_set_weights(dqn_handle *h, const float *weights);

/*
 * dqn_run -- one stream-ordered collection of N x L transitions.  Device
 * pointers, caller-owned:
 *   inputs   features [n_bars, 51] f32; starts [N] i32 (0 <= start,
 *            start + L <= n_bars - 1); seeds [N] u32 (LCG states)
 *   outputs  states [N, L, 54] f32; actions [N, L] i32; rewards [N, L] f32
 *            (curiosity bonus included); dones [N, L] i32; q [N, L] f32;
 *            td [N, L] f32; next_states [N, L, 54] f32 or NULL (the pre-reset
 *            next state of every transition)
 * 0 <= epsilon <= 1.  Validates everything checkable on the host first
 * (ROLLOUT_ERR_INVALID).  An out-of-range start zeroes that episode's outputs
 * and records ROLLOUT_ERR_RANGE; a device-side wait that times out records
 * ROLLOUT_ERR_TIMEOUT (read with dqn_status).  Step t of episode n reads bar
 * starts[n] + t, or with episode recycling on (dqn_set_recycle) the bar the
 * episode has moved to; states holds that bar's features.  The handle grows a
 * scratch array of N * L floats on the first call of a larger size
 * (ROLLOUT_ERR_NOMEM when that fails).  Returns ROLLOUT_OK, _INVALID, _NOMEM
 * or _CUDA.
 */
ROLLOUT_API int dqn_run(dqn_handle *h, const float *features, const int32_t *starts, const uint32_t *seeds, int N,
                        int L, float gamma, float epsilon, float *states, int32_t *actions, float *rewards,
                        int32_t *dones, float *q, float *td, float *next_states, void *stream);

/*
 * dqn_set_recycle -- episode recycling ("GPU Pipeline Phase 2b", section
 * "Future Phase 3 Optimization": an episode that ends starts again from a new
 * random bar instead of idling).  When on != 0, in every later dqn_run a done
 * at step t < L - 1 steps the episode's LCG state s once more and step t + 1
 * starts at bar ((s >> 8) * R) >> 24 with R = n_bars - L + t + 1 (every bar
 * that leaves room for the remaining steps and their next bars), with the
 * portfolio reset as on every done; the done transition's next state (in
 * next_states and behind td) stays the pre-reset state at the bar after its
 * own.  on == 0 (the default) continues the episode at the next bar.  The
 * handle then keeps an array of N * L int32 (the bar of every step), grown on
 * the first run of a larger size (ROLLOUT_ERR_NOMEM when that fails).  Returns
 * ROLLOUT_OK or ROLLOUT_ERR_INVALID (null handle).
 */
ROLLOUT_API int dqn_set_recycle(dqn_handle *h, int on);

/* dqn_set_timing -- on: later runs record CUDA events around their rollout,
 * state-row and target-pass kernels (for measurement).  dqn_phase_ms --
 * synchronises and writes the last timed run's three kernel times (ms).
 * Return ROLLOUT_OK, _INVALID (no timed run) or _CUDA. */
ROLLOUT_API int dqn_set_timing(dqn_handle *h, int on);
ROLLOUT_API int dqn_phase_ms(dqn_handle *h, float *ms);

/*
 * dqn_test_stall -- a test hook for the device-side timeout path, not for
 * production use.  When on != 0, every later dqn_run launches a test build of
 * the target pass in which CTA 0 never copies its first weight stage: that
 * CTA's MMA issuer waits on a stage that never fills, its bounded wait expires
 * after about two seconds, every warp of the CTA leaves, waits (bounded) for
 * its copies in flight and releases its tensor memory, and the run records
 * ROLLOUT_ERR_TIMEOUT (read with dqn_status).  The rollout and state-row
 * outputs (states, actions, dones, q) are complete; the rewards, td and
 * next_states of CTA 0's rows are then undefined.  on == 0 restores the
 * normal kernel.  Returns ROLLOUT_OK or ROLLOUT_ERR_INVALID (null handle).
 */
ROLLOUT_API int dqn_test_stall(dqn_handle *h, int on);

/* dqn_status -- synchronise the last stream used; ROLLOUT_OK or the first
 * device-side error since the last call (the word is then cleared). */
ROLLOUT_API int dqn_status(dqn_handle *h);

/* dqn_destroy -- frees the handle (NULL is a no-op); synchronises the device. */
ROLLOUT_API void dqn_destroy(dqn_handle *h);

#ifdef __cplusplus
}
#endif

#endif
