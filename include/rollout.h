/*
 * rollout.h -- C ABI of the GB300 (sm_103a) fused PPO experience collector.
 *
 * One call of rollout_run() collects N x L experience tuples with no host
 * round trip: N independent episodes each step through L bars.  Per step an
 * episode reads the 51 market features of its bar, appends 3 portfolio
 * features, runs the actor MLP 54->128->64->45 (ReLU), samples an action from
 * the softmax with a per-episode LCG uniform, runs the critic MLP
 * 54->512->384->256->128->64->1 (ReLU), and takes the portfolio,
 * triple-barrier, diversity-entropy and curiosity reward step, resetting the
 * episode on done.  A backward GAE scan per episode then produces advantages
 * and returns.
 *
 * Defining passages (page "PPO CUDA Pipeline Design -- Zero-Roundtrip
 * Experience Collection"): section "Kernel Phases", Phase A steps 1-12 (the
 * per-step body) and Phase B (GAE); section "Weight Layout" (tensor shapes and
 * the [out, in] row-major convention); section "Output Buffers" (outputs).
 * The environment functions it reuses are those of page "GPU Pipeline Phase
 * 2b: Zero-Roundtrip CUDA Experience Collection", section "Kernel Components".
 *
 * All entry points are thread-compatible, not thread-safe: calls that use the
 * same handle must not run concurrently (one stream, or external ordering).
 */
#ifndef ROLLOUT_H
#define ROLLOUT_H

#include <stdint.h>

#if defined(__GNUC__)
#define ROLLOUT_API __attribute__((visibility("default")))
#else
#define ROLLOUT_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* status codes (every entry point returns one of these, 0 = success) */
#define ROLLOUT_OK               0
#define ROLLOUT_ERR_INVALID     -1  /* null pointer, bad size, gamma/lambda outside [0,1] */
#define ROLLOUT_ERR_RANGE       -2  /* an episode start outside [0, n_bars - L - 1] (device-detected) */
#define ROLLOUT_ERR_CUDA        -3  /* a CUDA runtime call failed; see rollout_last_error() */
#define ROLLOUT_ERR_TIMEOUT     -4  /* a bounded device-side wait expired (device-detected) */
#define ROLLOUT_ERR_UNSUPPORTED -5  /* a network shape, dtype or constant the library does not handle */
#define ROLLOUT_ERR_NOMEM       -6  /* device allocation failed */

/* arithmetic of the MLPs (the environment, sampler and GAE are float32 throughout) */
#define ROLLOUT_FP32 0   /* float32 CUDA-core FMA */
#define ROLLOUT_TF32 1   /* tcgen05 kind::tf32 tensor cores, operands rounded to tf32 (ties away), f32 accumulate */
#define ROLLOUT_BF16 2   /* tcgen05 kind::f16 tensor cores, operands rounded to bf16 (nearest even), f32 accumulate */

/*
 * Network shapes, precision and environment constants, fixed at create time.
 * Supported shapes: n_market 51, n_actions 45, actor 128/64, curiosity 64,
 * critic hidden widths {512,384,256,128,64} or {1024,768,512,256,128}
 * (critic_nh = 5).  div_window in [1, 31].
 */
typedef struct {
    int   n_market;      /* market features per bar (51); state width is n_market + 3 */
    int   n_actions;     /* 45 = 5 exposures x 3 order types x 3 urgencies */
    int   actor_h1;      /* 128 */
    int   actor_h2;      /* 64 */
    int   critic_nh;     /* number of hidden critic layers (5) */
    int   critic_h[8];   /* their widths; the head is width 1 */
    int   cur_h;         /* curiosity hidden width (64) */
    int   dtype;         /* ROLLOUT_FP32 / ROLLOUT_TF32 / ROLLOUT_BF16 */
    int   n_bars;        /* rows of every features buffer passed to rollout_run */
    float barrier;       /* theta: done when portfolio PnL since reset >= +theta or <= -theta */
    int   max_hold;      /* K: done after K steps since reset */
    float pt_scale;      /* reward barrier_scale on a profit-take hit (0.5) */
    float sl_scale;      /* reward barrier_scale on a stop-loss hit (-0.5) */
    int   div_window;    /* diversity window length (20) */
    float div_thresh;    /* entropy threshold in bits (1.0) */
    float div_penalty;   /* added to the reward when entropy < threshold (-0.01) */
    float cur_coef;      /* curiosity bonus = cur_coef * MSE (0.01) */
    float risk_coef;     /* risk penalty = risk_coef * |exposure| (1e-3) */
    float tx_base;       /* cost rate = (1 + order + urgency) * tx_base (1e-4) */
    float spread;        /* third portfolio feature, a constant (1e-4) */
} rollout_dims;

typedef struct rollout_handle rollout_handle;

/*
 * rollout_create -- validate dims, convert and upload the weights.
 *
 * weights: HOST pointer to one packed float32 buffer, in this order, each
 *   matrix [out, in] row-major followed by its bias [out]:
 *     actor     W1[h1, n_market+3], b1, W2[h2, h1], b2, W3[n_actions, h2], b3
 *     critic    V1[c1, n_market+3], c1 ... V_nh[c_nh, c_nh-1], V_head[1, c_nh], head bias
 *     curiosity C1[cur_h, n_market+3+n_actions], d1, C2[n_market+3, cur_h], d2
 *   The library copies it (rounding to the dtype's operand format and
 *   re-tiling for the tensor cores); the caller keeps ownership and may free
 *   it on return.
 * out: receives the handle on success (unchanged on failure).
 * Allocates device memory on the current device; all later calls must use
 * that device.  The kernels' shared-memory limits are raised once on each
 * device that launches them, so handles on several devices of one process
 * work side by side.  Synchronous.  Returns ROLLOUT_OK, _INVALID,
 * _UNSUPPORTED, _NOMEM or _CUDA.
 */
ROLLOUT_API int rollout_create(const float *weights, const rollout_dims *dims, rollout_handle **out);

/*
 * rollout_set_weights -- replace the weights of an existing handle (same
 * packed layout as rollout_create; host pointer).  Synchronous with respect
 * to the host; runs already enqueued on a stream are ordered before it only
 * if the caller synchronises that stream first.
 */
ROLLOUT_API int rollout_set_weights(rollout_handle *h, const float *weights);

/*
 * rollout_set_weights_device -- rollout_set_weights from a DEVICE array of
 * the packed float32 weights (the layout rollout_create takes; for example a
 * PPO trainer's, see ppo.h), with no host round trip.  Enqueued on `stream`:
 * it rewrites the handle's converted weights element by element, rounding as
 * rollout_create does, so a later rollout_run on the same stream computes
 * what it would after rollout_set_weights with the same values.  `weights`
 * (caller-owned, 4-byte aligned) must stay valid until the work completes;
 * its values are not checked for finiteness, unlike rollout_set_weights.
 * Runs on the handle must be ordered after it (one stream, or an event).
 * (An addition of this library: the pages copy the updated weights from the
 * host.)  Returns ROLLOUT_OK, _INVALID or _CUDA.
 */
ROLLOUT_API int rollout_set_weights_device(rollout_handle *h, const float *weights, void *stream);

/*
 * rollout_run -- collect N x L experience tuples, including GAE.
 *
 * All array pointers are DEVICE pointers owned by the caller, 16-byte
 * aligned, on the handle's device:
 *   features        [n_bars, n_market] f32 row-major; column 0 is the bar's
 *                   log-return, so P[b+1]/P[b] = exp(features[b+1, 0])
 *   episode_starts  [N] i32, each in [0, n_bars - L - 1] (step t of episode n
 *                   uses bar start+t and reads bar start+t+1 for its return)
 *   seeds           [N] u32 initial LCG states; step t draws
 *                   s = s*1664525 + 1013904223 (mod 2^32), u = (s >> 8) * 2^-24
 *   out_states      [N, L, n_market+3] f32: [features of the bar, portfolio
 *                   value since reset, held exposure, spread]
 *   out_actions     [N, L] i32 in [0, n_actions)
 *   out_logp        [N, L] f32 log pi(action | state)
 *   out_values      [N, L] f32 critic value of the state
 *   out_rewards     [N, L] f32
 *   out_dones       [N, L] i32 (1 = the episode ended at this step and reset)
 *   out_adv         [N, L] f32 GAE advantages
 *   out_ret         [N, L] f32 returns = advantage + value
 * gamma, lambda: in [0, 1].  The bootstrap value after the last step is the
 *   critic of the last step's pre-reset next state.
 * stream: a cudaStream_t (NULL = legacy default stream).
 *
 * Stream-ordered and asynchronous: returns after enqueuing; every output is
 * fully overwritten by the time the stream reaches the end of the call (their
 * contents in between are unspecified -- some serve as intermediate storage).
 * Host-checkable arguments are validated before anything is enqueued
 * (ROLLOUT_ERR_INVALID); device-detected problems (an out-of-range start,
 * an expired bounded wait) are recorded in the handle's status word, read by
 * rollout_status().  An episode with an out-of-range start is not simulated
 * and its outputs are zero.  Returns ROLLOUT_OK, _INVALID or _CUDA.
 */
ROLLOUT_API int rollout_run(rollout_handle *h, const float *features, const int32_t *episode_starts,
                const uint32_t *seeds, int N, int L, float gamma, float lambda,
                float *out_states, int32_t *out_actions, float *out_logp, float *out_values,
                float *out_rewards, int32_t *out_dones, float *out_adv, float *out_ret,
                void *stream);

/*
 * rollout_status -- synchronise the stream of the last rollout_run on this
 * handle and return its device status: ROLLOUT_OK, ROLLOUT_ERR_RANGE or
 * ROLLOUT_ERR_TIMEOUT (or ROLLOUT_ERR_CUDA if the synchronisation failed).
 */
ROLLOUT_API int rollout_status(rollout_handle *h);

/*
 * rollout_set_timing -- when on != 0, every later rollout_run also records
 * CUDA events on its stream before and after each of its kernels (rollout,
 * state rows, value, GAE); off by default.  rollout_phase_ms synchronises the
 * last run's final event and writes the four kernels' device times in
 * milliseconds to ms[0..3].  Returns ROLLOUT_OK, _INVALID (timing was off or
 * no run yet) or _CUDA.
 */
ROLLOUT_API int rollout_set_timing(rollout_handle *h, int on);
ROLLOUT_API int rollout_phase_ms(rollout_handle *h, float *ms);

/*
 * rollout_test_stall -- a test hook for the device-side timeout path, not for
 * production use.  When on != 0, every later run of this handle on the
 * tensor-core path (ROLLOUT_TF32, ROLLOUT_BF16) launches a test build of the
 * value kernel in which CTA 0 never copies its first weight stage: that CTA's
 * MMA issuer waits on a stage that never fills, its bounded wait expires
 * after about two seconds, every warp of the CTA leaves, waits (bounded) for
 * its copies in flight and releases its tensor memory, and the run records
 * ROLLOUT_ERR_TIMEOUT (read with rollout_status).  The other CTAs finish
 * normally; the values, rewards, advantages and returns of CTA 0's tiles are
 * then undefined.  on == 0 restores the normal kernel.  Returns ROLLOUT_OK, or
 * ROLLOUT_ERR_INVALID for a null handle or an ROLLOUT_FP32 handle (whose
 * kernels have no waits).
 */
ROLLOUT_API int rollout_test_stall(rollout_handle *h, int on);

/*
 * rollout_forward -- the three networks on given states, for checking them in
 * isolation (test and debugging use, not the collection path).  Page "PPO
 * CUDA Pipeline Design -- Zero-Roundtrip Experience Collection", section
 * "Kernel Phases", Phase A steps 3 (actor: state -> logits), 5 (critic: state
 * -> value) and 9 (curiosity forward model: [state ; one-hot(action)] ->
 * predicted next state); section "Weight Layout".
 *
 * All arrays are DEVICE pointers owned by the caller, on the handle's device:
 *   states   [M, n_market+3] f32 (any values)
 *   actions  [M] i32 in [0, n_actions): the curiosity model's one-hot input
 *   logits   [M, n_actions] f32, values [M] f32, cur_pred [M, n_market+3] f32
 *            (outputs, fully overwritten)
 * The products run on the tensor cores in the handle's operand format, as
 * the collector's networks compute them: every weight and every layer input
 * rounded once to bf16 (ROLLOUT_BF16) or tf32 (ROLLOUT_TF32), float32
 * accumulation, float32 bias and ReLU; ROLLOUT_FP32 handles take float32-grade
 * products (each operand split into three bf16 parts, the six largest
 * products of parts taken: relative error below 2^-22 per product).  The handle
 * keeps a device copy of the float32 weights for this (refreshed by
 * rollout_set_weights and rollout_set_weights_device) and its own buffers,
 * grown on demand.  Stream-ordered and asynchronous.  An action out of range
 * gives a zero one-hot and records ROLLOUT_ERR_RANGE in the status word
 * (rollout_status).  Returns ROLLOUT_OK, _INVALID, _NOMEM or _CUDA.
 */
ROLLOUT_API int rollout_forward(rollout_handle *h, const float *states, const int32_t *actions, int M,
                                float *logits, float *values, float *cur_pred, void *stream);

/*
 * rollout_test_activations -- a test hook for checking the tensor-core paths
 * layer by layer, not for production use.  (An addition of this library: the
 * page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
 * section "Kernel Phases", Phase A steps 3, 5 and 9, defines the actor, critic
 * and curiosity networks whose hidden layers it exposes.)
 *
 * When dump != NULL, every later run of this handle on the tensor-core path
 * (ROLLOUT_TF32, ROLLOUT_BF16) launches test builds of the rollout and value
 * kernels that also write, for episodes 0..n_episodes-1, every operand its
 * layers consumed: the state input and each hidden activation (after bias,
 * ReLU and rounding to the operand format: a bf16 or tf32 value, stored as
 * float32).
 * dump: DEVICE array, caller-owned, 16-byte aligned, of
 *   n_episodes * (L + 1) rows of W floats, W = 64 + actor_h1 + actor_h2 +
 *   (sum of the critic hidden widths) + cur_h (1664 for the standard critic,
 *   3008 for the widened one).  Row n*(L+1) + t is step t of episode n:
 *   [state input (64 columns, the first n_market + 3 written) | actor h1 |
 *   actor h2 | critic hidden layers 1..critic_nh | curiosity hidden]; row
 *   n*(L+1) + L is episode n's bootstrap critic (its state input and critic
 *   columns only).  Columns a run does not produce are left as they were.
 *   Episodes at or beyond the run's N are not written.  The array must stay
 *   valid while runs that use it are in flight.
 * dump == NULL restores the normal kernels (the timed kernels never write
 * it).  The other outputs of a dumping run equal those of a normal run.
 * Returns ROLLOUT_OK, or ROLLOUT_ERR_INVALID for a null handle, an
 * ROLLOUT_FP32 handle (nothing is rounded), n_episodes <= 0 or a misaligned
 * array.
 */
ROLLOUT_API int rollout_test_activations(rollout_handle *h, float *dump, int n_episodes);

/*
 * rollout_test_alloc -- a test hook for allocation failures, not for
 * production use.  (An addition of this library; the pages name no such
 * hook.)  Every device allocation that a rollout handle makes (in
 * rollout_create, rollout_set_weights and rollout_run_host's staging) is
 * counted.  After rollout_test_alloc(k, ...) with k > 0, the k-th such
 * allocation fails as if the device were out of memory; the call that
 * needed it then returns ROLLOUT_ERR_NOMEM after freeing whatever it had
 * allocated.  k <= 0 turns the hook off.  Every call restarts the count.
 * live (may be NULL) receives the number of the library's device allocations
 * currently held.  Process-wide; not thread-safe with respect to concurrent
 * creates.  Returns ROLLOUT_OK.
 */
ROLLOUT_API int rollout_test_alloc(long long fail_at, long long *live);

/*
 * rollout_run_static -- rollout_run for callers that cannot allocate device
 * memory.  (An addition of this library; the paper has no counterpart.)
 *
 * Who needs it: code that must not call cudaMalloc -- a path that runs while
 * a CUDA graph is being captured, a latency-critical loop that must never
 * block on the device allocator, or a host that hands the library a fixed
 * device-memory budget at start-up and forbids later allocations.  The tf32
 * and widened-critic configurations run their value phase with per-CTA
 * activation scratch; rollout_run takes it from memory rollout_create
 * allocated, this entry point takes it from a fixed array compiled into the
 * library (ROLLOUT_STATIC_SCRATCH_BYTES, 16 MiB), and it allocates nothing
 * itself.  Every GPU that loads the library holds that array until the
 * process exits.  Other configurations use no scratch and run exactly as
 * rollout_run.
 *
 * Same arguments, results, stream ordering and return codes as
 * rollout_run, plus ROLLOUT_ERR_UNSUPPORTED when the handle's layer shapes
 * need more scratch per CTA than the array holds.  The value phase then runs
 * on at most ROLLOUT_STATIC_SCRATCH_BYTES / (scratch per CTA) CTAs, so it is
 * slower than rollout_run for large batches.
 *
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) and caches it; make that first call before any
 * stream capture on that device.  All calls share the one array, which keeps
 * the last call's contents (nothing in it has to start at zero: every tile
 * writes its activations before reading them): calls that overlap on the
 * GPU -- on different streams, handles or host threads -- race on it and
 * must be serialised by the caller.
 */
#define ROLLOUT_STATIC_SCRATCH_BYTES (16u << 20)
ROLLOUT_API int rollout_run_static(rollout_handle *h, const float *features, const int32_t *episode_starts,
                                   const uint32_t *seeds, int N, int L, float gamma, float lambda,
                                   float *out_states, int32_t *out_actions, float *out_logp, float *out_values,
                                   float *out_rewards, int32_t *out_dones, float *out_adv, float *out_ret,
                                   void *stream);

/*
 * rollout_run_host -- rollout_run from and to HOST memory.  (An addition of
 * this library: the pages' pipeline downloads six output buffers after its
 * kernel -- page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience
 * Collection", section "Output Buffers"; here every download starts as soon
 * as the kernel that finishes that output is done.)
 *
 * features, episode_starts, seeds: HOST arrays with the layouts rollout_run
 * gives (features is [n_bars, n_market], the handle's n_bars).  The out_*
 * arrays are HOST arrays with rollout_run's layouts; any of them may be NULL,
 * and that output is then not copied back.  No alignment is required.
 *
 * The inputs are copied to device memory that the handle owns and keeps for
 * later calls: the first call, and any call with a larger N * L, allocates it
 * (about 4 * N * L * (n_market + 10) + 4 * n_bars * n_market bytes) and
 * waits for the device if it has to free a smaller one.  The kernels then
 * run as in rollout_run, and each output is copied back on one of the
 * handle's four copy streams right after its kernel: actions, log-probs and
 * dones after the rollout, the state rows after the state-row kernel (while
 * the value kernel runs), values and rewards after the value kernel,
 * advantages and returns after GAE.  Outputs above 64 MiB are split over the
 * four streams.  `stream` waits for every copy at the end, so the call is
 * stream-ordered like rollout_run: once the stream has reached the end of the
 * call, the host outputs hold the results.  Copies only overlap the kernels
 * when the host arrays are page-locked (cudaHostAlloc / cudaHostRegister);
 * with pageable memory the call returns only after those copies are done.
 *
 * Returns ROLLOUT_OK, _INVALID, _NOMEM or _CUDA; device-detected problems go
 * to rollout_status() as for rollout_run.  Calls on one handle must be
 * ordered (one stream, or external synchronisation): they share the device
 * copies.
 */
ROLLOUT_API int rollout_run_host(rollout_handle *h, const float *features, const int32_t *episode_starts,
                                 const uint32_t *seeds, int N, int L, float gamma, float lambda,
                                 float *out_states, int32_t *out_actions, float *out_logp, float *out_values,
                                 float *out_rewards, int32_t *out_dones, float *out_adv, float *out_ret,
                                 void *stream);

/* rollout_destroy -- free the handle and its device memory (NULL is a no-op).
 * Synchronises the device first. */
ROLLOUT_API void rollout_destroy(rollout_handle *h);

/* rollout_last_error -- message of the last failed call on this host thread
 * ("" if none).  The pointer stays valid until the next call on the thread. */
ROLLOUT_API const char *rollout_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* ROLLOUT_H */
