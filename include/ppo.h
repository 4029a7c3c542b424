/*
 * ppo.h -- C ABI of the on-device PPO update that consumes the tuples
 * rollout_run collected, without them leaving the GPU.
 *
 * Defining passages: page "PPO CUDA Pipeline Design -- Zero-Roundtrip
 * Experience Collection", the training flow after the collector (for each PPO
 * epoch, for each mini-batch: recompute log-probs through the actor, ratio =
 * exp(new - old), PPO clipped surrogate loss plus critic MSE loss, backward,
 * optimizer step); page "Fused CUDA Training Kernel -- Implementation Plan",
 * "Chunk 3: Adam Optimizer Kernel" (gradient L2 norm, clip scale
 * min(max_norm / (norm + eps), 1), bias-corrected Adam with a decoupled
 * weight-decay term).
 *
 * The loss of a mini-batch of B tuples i (advantage A_i, return R_i, old
 * log-prob lo_i, ratio rho_i = exp(log pi(a_i|s_i) - lo_i), critic value v_i):
 *   L = -(1/B) sum_i min(rho_i A_i, clip(rho_i, 1-eps, 1+eps) A_i)
 *       + value_coef (1/B) sum_i (v_i - R_i)^2
 * Where both surrogate terms are equal the unclipped one carries the
 * gradient; ReLU'(0) = 0.  The gradient over the actor and the critic together
 * is scaled by min(1, max_grad_norm / (|g| + 1e-6)) (no scaling when
 * max_grad_norm <= 0), then one Adam step (moments from zero, bias
 * correction with the step count t = 1, 2, ...) updates both:
 *   m = b1 m + (1-b1) g;  v = b2 v + (1-b2) g^2;
 *   p -= lr (m / (1-b1^t)) / (sqrt(v / (1-b2^t)) + adam_eps) + weight_decay p.
 * The curiosity weights are not trained.  Parameters, gradients and Adam
 * moments are float32; the dense layers run as float32 GEMMs (cuBLAS, no
 * reduced-precision math) and everything else in this library's kernels.
 *
 * Thread-compatible, not thread-safe: calls on one trainer must be ordered.
 */
#ifndef PPO_H
#define PPO_H

#include <stdint.h>

#include "rollout.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct ppo_trainer ppo_trainer;

typedef struct {
    float clip_eps;        /* 0.2 */
    float value_coef;      /* 1.0 */
    float lr;              /* 3e-4 */
    float beta1, beta2;    /* 0.9, 0.999 */
    float adam_eps;        /* 1e-8 */
    float max_grad_norm;   /* 0.5; <= 0: no clipping */
    float weight_decay;    /* 0 */
} ppo_hparams;

/*
 * ppo_create -- a trainer over a float32 copy (device, trainer-owned) of the
 * packed weights (the layout rollout_create takes), with zero Adam state.
 * dims gives the network shapes (dtype is ignored: the update is float32).
 * Returns ROLLOUT_OK, _INVALID, _UNSUPPORTED (a shape rollout_create would
 * refuse), _NOMEM or _CUDA.
 */
ROLLOUT_API int ppo_create(const float *weights, const rollout_dims *dims, ppo_trainer **out);

/*
 * ppo_update -- n_steps optimizer steps on `stream`.  Step k uses the
 * mini-batch of tuples indices[k*batch .. k*batch + batch).
 * All arrays are DEVICE pointers owned by the caller, the tuple arrays as
 * rollout_run writes them, flattened over (episode, step):
 *   states   [T, n_market+3] f32     actions  [T] i32 in [0, n_actions)
 *   logp_old [T] f32                 adv, ret [T] f32
 *   indices  [n_steps * batch] i32, each in [0, T)
 *   stats    [n_steps, 5] f32 or NULL: per step the surrogate loss, the value
 *            loss (before value_coef), the fraction of rows whose clipped term
 *            was the smaller, the mean ratio, and the gradient norm before
 *            clipping.
 * batch in [1, 4096].  Stream-ordered and asynchronous.  An index out of
 * range is replaced by 0 and recorded in the trainer's status word
 * (ppo_status: ROLLOUT_ERR_RANGE).  Returns ROLLOUT_OK, _INVALID, _NOMEM
 * (the first call, or a larger batch, allocates the mini-batch buffers) or
 * _CUDA.
 */
ROLLOUT_API int ppo_update(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                           const float *adv, const float *ret, long long T, const int32_t *indices, int n_steps,
                           int batch, const ppo_hparams *hp, float *stats, void *stream);

/*
 * ppo_gradient -- the loss statistics and the gradient of one mini-batch
 * (indices[0 .. batch)) at the current weights, without an optimizer step:
 * grad receives the n_trained = actor + critic parameters' gradient
 * (float32, packed layout order, before any clipping), stats (4 floats or
 * NULL) the first four per-step statistics of ppo_update.  For gradient
 * checks and gradient accumulation.  Arguments and return codes otherwise
 * as ppo_update.
 */
ROLLOUT_API int ppo_gradient(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                             const float *adv, const float *ret, long long T, const int32_t *indices, int batch,
                             const ppo_hparams *hp, float *grad, float *stats, void *stream);

/*
 * ppo_test_activations -- a test hook (not for production use): copies the
 * hidden activations of the last mini-batch forward pass (that of the last
 * ppo_gradient call, or of the last step of ppo_update) to `act` (device or
 * host), after the work enqueued on `stream`: row r of the batch is
 * [actor hidden layers | critic hidden layers] (actor_h1 + actor_h2 + the
 * critic's hidden widths floats, after the ReLU).  Lets a check see which side
 * of the ReLU kink the float32 tensor-core products put each pre-activation.
 * (An addition of this library: page "Fused CUDA Training Kernel --
 * Implementation Plan", "Chunk 2: Backward Pass Kernel", defines the masks it
 * exposes.)  Returns ROLLOUT_OK, _INVALID (no forward pass yet) or _CUDA.
 */
ROLLOUT_API int ppo_test_activations(ppo_trainer *t, float *act, void *stream);

/* ppo_get_weights -- copy the packed float32 weights (device or host
 * destination, n_weights floats) after the work enqueued on `stream`. */
ROLLOUT_API int ppo_get_weights(ppo_trainer *t, float *weights, void *stream);

/* ppo_device_weights -- the trainer's own device array of the packed float32
 * weights (n_weights floats), which ppo_update rewrites in place; valid until
 * ppo_destroy.  Pass it to rollout_set_weights_device, on the stream of the
 * updates, to refresh a rollout handle with no copy. */
ROLLOUT_API int ppo_device_weights(ppo_trainer *t, const float **weights);

/* ppo_reset_optimizer -- zero the Adam moments and the step count (on `stream`). */
ROLLOUT_API int ppo_reset_optimizer(ppo_trainer *t, void *stream);

/* ppo_status -- synchronise the last stream used and return ROLLOUT_OK or
 * ROLLOUT_ERR_RANGE (an index was out of range since the last call). */
ROLLOUT_API int ppo_status(ppo_trainer *t);

/* ppo_destroy -- free the trainer (NULL is a no-op).  Synchronises the device. */
ROLLOUT_API void ppo_destroy(ppo_trainer *t);

#ifdef __cplusplus
}
#endif

#endif
