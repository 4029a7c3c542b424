/*
 * per.h -- C ABI of the GPU-resident prioritised experience replay buffer:
 * a fixed-capacity ring of transitions and their priorities in device
 * memory, proportional sampling with importance-sampling weights, and the
 * priority scatter after a training step, all stream-ordered with no host
 * synchronisation.
 *
 * Defining passages: page "GPU-Resident Prioritized Experience Replay",
 * sections "New struct: GpuReplayBuffer" (the ring's arrays; write cursor and
 * size kept on the host), "Sampling Kernels / Proportional" (uniforms in
 * [0, total), cumulative priorities, a binary search per sample, gather, IS
 * weights (1 / (N p_i / total))^beta / max weight), "Priority update" (priority
 * = |td|^alpha + epsilon, scattered to the sampled slots), "Experience
 * Insertion" (device-to-device copies; new transitions get the maximum
 * priority; the cursor wraps) and "Error Handling" (non-finite priorities
 * clamped into [epsilon, max priority]).
 *
 * Definitions (size = number of stored transitions, p the priorities of slots
 * 0 .. size-1, total = sum p, c_i = p_0 + ... + p_i):
 *   sample k draws u_k in [0, 1) (below), t_k = u_k total (moved just below
 *     total if the product rounds up to it), and picks the slot
 *     i_k = min { i : c_i > t_k }  (a slot of zero priority is never picked);
 *   its weight is w_k = (size p_{i_k} / total)^(-beta) / max_j w_j (max over
 *     the batch), formed in float32 (x = size p / total, 2^(-beta log2 x), the
 *     division by the maximum): within about (5 + 1.5 beta |log2 x|) 2^-24
 *     relative of the exact value;
 *   u_k = (x >> 11) 2^-53 with x the (offset + k)-th output (counting from 0)
 *     of the SplitMix64 generator seeded with `seed` (Steele, Lea & Flood,
 *     OOPSLA 2014): x = mix(seed + (offset + k + 1) 0x9E3779B97F4A7C15);
 *   an update sets p_i = fl32(|td|^alpha + eps) (computed in double, rounded
 *     once to float32) for each slot i it names; where a batch names a slot
 *     more than once the last entry wins; a NaN td gives eps and a priority
 *     past float32 (+inf) the maximum priority held before the call;
 *   the maximum priority starts at 1 and is the running maximum of every
 *     priority an update has written (it never decreases); inserted
 *     transitions take it.
 * Sums run in double; the sample's slot is the exact-arithmetic answer except
 * where t_k lies within rounding (about 1e-12 total) of a boundary c_i.
 *
 * Thread-compatible, not thread-safe: calls on one buffer must be ordered
 * (one stream, or events).  Status codes are rollout.h's.
 */
#ifndef PER_H
#define PER_H

#include <stdint.h>

#include "rollout.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct per_buffer per_buffer;

/*
 * per_create -- a buffer of `capacity` transitions (1 <= capacity < 2^31) of
 * `state_dim`-float states (1 <= state_dim <= 4096), empty, maximum priority 1.
 * Allocates every device array once (about capacity * (8 state_dim + 21)
 * bytes).  Returns ROLLOUT_OK, _INVALID, _NOMEM or _CUDA.
 */
ROLLOUT_API int per_create(long long capacity, int state_dim, per_buffer **out);

/*
 * per_insert -- append `count` transitions (device pointers, caller-owned):
 *   states, next_states [count, state_dim] f32; actions [count] i32;
 *   rewards [count] f32; dones [count] u8.
 * Transition j goes to slot (cursor + j) mod capacity, as if inserted one at a
 * time (when count > capacity only the last `capacity` survive); each gets the
 * current maximum priority.  The cursor and size advance on the host.
 * Enqueued on `stream`.  Returns ROLLOUT_OK, _INVALID or _CUDA.
 */
ROLLOUT_API int per_insert(per_buffer *b, const float *states, const float *next_states, const int32_t *actions,
                           const float *rewards, const uint8_t *dones, long long count, void *stream);

/*
 * per_sample -- draw `batch` transitions (1 <= batch <= 65536) as defined
 * above and gather them.  Outputs are device pointers, caller-owned:
 *   indices [batch] i32; is_weights [batch] f32;
 *   states, next_states [batch, state_dim] f32; actions [batch] i32;
 *   rewards [batch] f32; dones [batch] u8  (any gathered output may be NULL).
 * Enqueued on `stream`.  A buffer whose priorities sum to zero records
 * ROLLOUT_ERR_RANGE in the status word and returns slot 0 with weight 0.
 * Returns ROLLOUT_OK, _INVALID (empty buffer, bad batch or beta) or _CUDA.
 */
ROLLOUT_API int per_sample(per_buffer *b, int batch, float beta, uint64_t seed, uint64_t offset, int32_t *indices,
                           float *is_weights, float *states, float *next_states, int32_t *actions, float *rewards,
                           uint8_t *dones, void *stream);

/*
 * per_update_priorities -- p_i = |td_k|^alpha + eps for slot i = indices[k],
 * k < batch (device arrays: indices i32, td_errors f32), as defined above.
 * alpha >= 0, eps >= 0.  A slot outside [0, size) is skipped and recorded
 * (ROLLOUT_ERR_RANGE).  Enqueued on `stream`.  Returns ROLLOUT_OK, _INVALID or
 * _CUDA.
 */
ROLLOUT_API int per_update_priorities(per_buffer *b, const int32_t *indices, const float *td_errors, int batch,
                                      float alpha, float eps, void *stream);

/* per_size -- the number of stored transitions and the write cursor (host values). */
ROLLOUT_API int per_size(per_buffer *b, long long *size, long long *cursor);

/* per_read -- copy the priorities [capacity] f32 and the maximum priority (1
 * float) to `priorities` / `max_priority` (device or host, either may be NULL)
 * after the work enqueued on `stream`; for checks and checkpoints. */
ROLLOUT_API int per_read(per_buffer *b, float *priorities, float *max_priority, void *stream);

/* per_status -- synchronise the last stream used and return ROLLOUT_OK or
 * ROLLOUT_ERR_RANGE (an update named a slot out of range, or a sample met a
 * zero total, since the last call); the status word is cleared. */
ROLLOUT_API int per_status(per_buffer *b);

/* per_destroy -- free the buffer (NULL is a no-op).  Synchronises the device. */
ROLLOUT_API void per_destroy(per_buffer *b);

#ifdef __cplusplus
}
#endif

#endif
