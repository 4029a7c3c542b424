/*
 * ppo.c -- plain, slow, single-threaded CPU statement of the PPO update that
 * consumes the collected tuples: per mini-batch, the actor's log-probabilities
 * are recomputed, the clipped surrogate and the critic's squared error are
 * formed, their gradient is taken by backpropagation, clipped to a global
 * L2 norm and applied by one Adam step.  All arithmetic is in double.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests and the benchmark's CPU baseline do.  It
 * shares no code, header, table or constant with the CUDA path.
 *
 * Source: page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience
 * Collection", the training flow after the collector: for each PPO epoch, for
 * each mini-batch, recompute log-probs through the actor, ratio =
 * exp(new log-prob - old log-prob), PPO clipped surrogate loss plus critic MSE
 * loss, backward and an optimizer step; and page "Fused CUDA Training Kernel --
 * Implementation Plan", "Chunk 3: Adam Optimizer Kernel" (gradient L2 norm,
 * scale = min(max_norm / (norm + eps), 1), then per element the Adam update
 * with bias correction and a decoupled weight-decay term wd * param).
 *
 * Readings where the pages are silent (listed with their reasons in the
 * design notes): the loss of a mini-batch of B rows is
 *   L = -(1/B) sum_i min(rho_i A_i, clip(rho_i, 1-eps, 1+eps) A_i)
 *       + c_v (1/B) sum_i (v_i - R_i)^2
 * with A the GAE advantage and R the return, no entropy term and no
 * advantage normalisation; where both surrogate terms are equal the
 * unclipped one carries the gradient; ReLU'(0) = 0; one Adam state covers the
 * actor and the critic; the norm's eps is 1e-6 and |g| is taken over actor
 * and critic together; Adam's moments start at zero and are bias-corrected
 * with the step count t (1, 2, ...).  The curiosity weights in the packed
 * vector are left as they are.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define PPO_MAX_W 1024
#define PPO_MAX_LAYERS 8

typedef struct {
    int n_market, n_actions, actor_h1, actor_h2, critic_nh;
    int critic_h[8];
    int cur_h;
} ppo_shape;

typedef struct {
    double clip_eps, value_coef, lr, beta1, beta2, adam_eps, max_grad_norm, weight_decay;
} ppo_hp;

/* offsets of the dense layers in the packed weight vector ([out, in] row-major
 * matrix, then its bias; actor, critic, curiosity) */
typedef struct {
    int n_layers;
    long w[PPO_MAX_LAYERS], b[PPO_MAX_LAYERS];
    int in[PPO_MAX_LAYERS], out[PPO_MAX_LAYERS];
} net;

static long layout(const ppo_shape *s, net *actor, net *critic)
{
    long off = 0;
    const int sd = s->n_market + 3;
    const int ai[3] = {sd, s->actor_h1, s->actor_h2}, ao[3] = {s->actor_h1, s->actor_h2, s->n_actions};
    actor->n_layers = 3;
    for (int l = 0; l < 3; ++l) {
        actor->in[l] = ai[l];
        actor->out[l] = ao[l];
        actor->w[l] = off; off += (long)ai[l] * ao[l];
        actor->b[l] = off; off += ao[l];
    }
    critic->n_layers = s->critic_nh + 1;
    int prev = sd;
    for (int l = 0; l < critic->n_layers; ++l) {
        const int o = l < s->critic_nh ? s->critic_h[l] : 1;
        critic->in[l] = prev;
        critic->out[l] = o;
        critic->w[l] = off; off += (long)prev * o;
        critic->b[l] = off; off += o;
        prev = o;
    }
    return off;   /* end of the critic: the trained parameters are [0, off) */
}

long ppo_trained_count(const ppo_shape *s)
{
    net a, c;
    return layout(s, &a, &c);
}

/* Replay of the path's ReLU decisions.  The path under test computes each
 * hidden pre-activation z in float32 from products whose relative error is at
 * most 2^-15 (its operands' split), so where the exact z lies within
 * (2^-15 + (K + 4) 2^-23) sum|terms| of 0 it may take the other side of the
 * kink: a floating-point decision, like an action drawn within rounding of a
 * CDF boundary.  There the oracle adopts the path's activation (a replay);
 * a different side farther from the kink is a mismatch (adopted as well). */
typedef struct {
    long replays, mismatches;
} ppo_replay;

/* forward pass keeping every layer's output: act[l] is layer l's output
 * (after the ReLU for hidden layers), act_in = the input.  gact (or NULL):
 * the path's hidden activations of this row and net, layer after layer,
 * replayed as above. */
static void forward(const double *p, const net *n, const double *x, double act[][PPO_MAX_W], const float *gact,
                    ppo_replay *rp)
{
    const double *in = x;
    long at = 0;
    for (int l = 0; l < n->n_layers; ++l) {
        const int last = l == n->n_layers - 1;
        for (int j = 0; j < n->out[l]; ++j) {
            double acc = p[n->b[l] + j], mag = fabs(p[n->b[l] + j]);
            for (int i = 0; i < n->in[l]; ++i) {
                const double t = p[n->w[l] + (long)j * n->in[l] + i] * in[i];
                acc += t;
                mag += fabs(t);
            }
            double y = (!last && acc <= 0.0) ? 0.0 : acc;
            if (gact && !last) {
                const double g = (double)gact[at + j];
                if ((g > 0.0) != (acc > 0.0)) {
                    const double bound = (ldexp(1.0, -15) + (double)(n->in[l] + 4) * ldexp(1.0, -23)) * mag;
                    if (fabs(acc) <= bound) rp->replays++;
                    else rp->mismatches++;
                    y = g > 0.0 ? g : 0.0;
                }
            }
            act[l][j] = y;
        }
        if (!last) at += n->out[l];
        in = act[l];
    }
}

/* backpropagation of dout (gradient at the network's output) through n,
 * accumulating into the gradient vector g (same layout as p) */
static void backward(const double *p, const net *n, const double *x, double act[][PPO_MAX_W],
                     const double *dout, double *g)
{
    double d[PPO_MAX_W], dprev[PPO_MAX_W];
    const int L = n->n_layers;
    memcpy(d, dout, sizeof(double) * n->out[L - 1]);
    for (int l = L - 1; l >= 0; --l) {
        const double *in = l == 0 ? x : act[l - 1];
        for (int j = 0; j < n->out[l]; ++j) {
            g[n->b[l] + j] += d[j];
            for (int i = 0; i < n->in[l]; ++i) g[n->w[l] + (long)j * n->in[l] + i] += d[j] * in[i];
        }
        if (l == 0) break;
        for (int i = 0; i < n->in[l]; ++i) {
            double acc = 0.0;
            for (int j = 0; j < n->out[l]; ++j) acc += p[n->w[l] + (long)j * n->in[l] + i] * d[j];
            dprev[i] = act[l - 1][i] > 0.0 ? acc : 0.0;   /* ReLU' of the layer below, 0 at 0 */
        }
        memcpy(d, dprev, sizeof(double) * n->in[l]);
    }
}

/*
 * The smallest relative distance of any hidden pre-activation of the actor and
 * the critic from the ReLU kink on each row: margin[i] = min over hidden units
 * of |pre| / (|b| + sum |w x|).  Where it is of the order of float32 rounding,
 * a float32 evaluation may take the other side of the kink (a floating-point
 * decision, like an action drawn within rounding of a CDF boundary), and that
 * row's gradient through every earlier layer changes with it.
 */
void ppo_kink_margin(const double *p, const ppo_shape *s, const float *states, const int32_t *rows, int B,
                     double *margin)
{
    net an, cn;
    layout(s, &an, &cn);
    const int sd = s->n_market + 3;
    double in[PPO_MAX_W], out[PPO_MAX_W];
    const net *nets[2] = {&an, &cn};
    for (int r = 0; r < B; ++r) {
        double best = INFINITY;
        for (int k = 0; k < 2; ++k) {
            const net *n = nets[k];
            for (int i = 0; i < sd; ++i) in[i] = (double)states[(long)rows[r] * sd + i];
            for (int l = 0; l < n->n_layers - 1; ++l) {
                for (int j = 0; j < n->out[l]; ++j) {
                    double acc = p[n->b[l] + j], mag = fabs(p[n->b[l] + j]);
                    for (int i = 0; i < n->in[l]; ++i) {
                        const double t = p[n->w[l] + (long)j * n->in[l] + i] * in[i];
                        acc += t;
                        mag += fabs(t);
                    }
                    if (mag > 0.0 && fabs(acc) / mag < best) best = fabs(acc) / mag;
                    out[j] = acc <= 0.0 ? 0.0 : acc;
                }
                memcpy(in, out, sizeof(double) * n->out[l]);
            }
        }
        margin[r] = best;
    }
}

/*
 * Loss and gradient of one mini-batch.  rows[i] indexes the tuple arrays
 * (states [T, n_market+3], actions, logp_old, adv, ret).  g (length
 * ppo_trained_count) is overwritten.  stats (optional): [0] surrogate loss,
 * [1] value loss (before c_v), [2] fraction of rows whose clipped term is the
 * smaller, [3] mean ratio.
 */
void ppo_loss_grad_replay(const double *p, const ppo_shape *s, const ppo_hp *hp, const float *states,
                          const int32_t *actions, const float *logp_old, const float *adv, const float *ret,
                          const int32_t *rows, int B, double *g, double *stats, const float *gpu_act, long gpu_ld,
                          long *replays, long *mismatches);

void ppo_loss_grad(const double *p, const ppo_shape *s, const ppo_hp *hp, const float *states,
                   const int32_t *actions, const float *logp_old, const float *adv, const float *ret,
                   const int32_t *rows, int B, double *g, double *stats)
{
    ppo_loss_grad_replay(p, s, hp, states, actions, logp_old, adv, ret, rows, B, g, stats, NULL, 0, NULL, NULL);
}

/* ppo_loss_grad, given the path's hidden activations of the mini-batch
 * (gpu_act row r at gpu_act + r * gpu_ld: [actor hidden layers | critic
 * hidden layers]), replaying its ReLU decisions (see ppo_replay); the counts
 * go to *replays and *mismatches. */
void ppo_loss_grad_replay(const double *p, const ppo_shape *s, const ppo_hp *hp, const float *states,
                          const int32_t *actions, const float *logp_old, const float *adv, const float *ret,
                          const int32_t *rows, int B, double *g, double *stats, const float *gpu_act, long gpu_ld,
                          long *replays, long *mismatches)
{
    ppo_replay rp = {0, 0};
    net an, cn;
    const long np = layout(s, &an, &cn);
    const int sd = s->n_market + 3, na = s->n_actions;
    double act[PPO_MAX_LAYERS][PPO_MAX_W];
    double x[PPO_MAX_W], dl[PPO_MAX_W];
    memset(g, 0, sizeof(double) * np);
    double l_clip = 0.0, l_v = 0.0, n_clipped = 0.0, sum_rho = 0.0;
    for (int r = 0; r < B; ++r) {
        const long row = rows[r];
        for (int i = 0; i < sd; ++i) x[i] = (double)states[row * sd + i];
        const int a = actions[row];
        const double A = (double)adv[row], R = (double)ret[row];
        const float *ga = gpu_act ? gpu_act + (long)r * gpu_ld : NULL;
        /* actor: log-softmax of the taken action */
        forward(p, &an, x, act, ga, &rp);
        const double *lg = act[an.n_layers - 1];
        double m = lg[0];
        for (int j = 1; j < na; ++j) m = lg[j] > m ? lg[j] : m;
        double z = 0.0;
        for (int j = 0; j < na; ++j) z += exp(lg[j] - m);
        const double logp = (lg[a] - m) - log(z);
        const double rho = exp(logp - (double)logp_old[row]);
        const double rc = rho < 1.0 - hp->clip_eps ? 1.0 - hp->clip_eps : (rho > 1.0 + hp->clip_eps ? 1.0 + hp->clip_eps : rho);
        const double s1 = rho * A, s2 = rc * A;
        const int unclipped = s1 <= s2;
        l_clip += -(unclipped ? s1 : s2);
        n_clipped += unclipped ? 0.0 : 1.0;
        sum_rho += rho;
        /* d L / d logp = -A rho / B on the unclipped branch, 0 on the clipped one */
        const double glp = unclipped ? -A * rho / (double)B : 0.0;
        for (int j = 0; j < na; ++j) dl[j] = glp * ((j == a ? 1.0 : 0.0) - exp(lg[j] - m) / z);
        backward(p, &an, x, act, dl, g);
        /* critic */
        forward(p, &cn, x, act, ga ? ga + s->actor_h1 + s->actor_h2 : NULL, &rp);
        const double v = act[cn.n_layers - 1][0];
        l_v += (v - R) * (v - R);
        const double dv = 2.0 * hp->value_coef * (v - R) / (double)B;
        backward(p, &cn, x, act, &dv, g);
    }
    if (replays) *replays = rp.replays;
    if (mismatches) *mismatches = rp.mismatches;
    if (stats) {
        stats[0] = l_clip / B;
        stats[1] = l_v / B;
        stats[2] = n_clipped / B;
        stats[3] = sum_rho / B;
    }
}

/* global-norm clipping and one Adam step (t = the step's count, from 1);
 * returns the gradient norm before clipping */
double ppo_adam_step(double *p, double *g, double *m, double *v, long n, long t, const ppo_hp *hp)
{
    double ss = 0.0;
    for (long i = 0; i < n; ++i) ss += g[i] * g[i];
    const double norm = sqrt(ss);
    double scale = 1.0;
    if (hp->max_grad_norm > 0.0) {
        const double c = hp->max_grad_norm / (norm + 1e-6);
        scale = c < 1.0 ? c : 1.0;
    }
    const double bc1 = 1.0 - pow(hp->beta1, (double)t), bc2 = 1.0 - pow(hp->beta2, (double)t);
    for (long i = 0; i < n; ++i) {
        const double gi = g[i] * scale;
        m[i] = hp->beta1 * m[i] + (1.0 - hp->beta1) * gi;
        v[i] = hp->beta2 * v[i] + (1.0 - hp->beta2) * gi * gi;
        p[i] -= hp->lr * (m[i] / bc1) / (sqrt(v[i] / bc2) + hp->adam_eps) + hp->weight_decay * p[i];
    }
    return norm;
}

/*
 * n_steps optimizer steps; step k uses rows[k*B .. k*B+B).  w (packed float32
 * weights, actor and critic updated in place, rounded to float32 after the
 * last step) and the Adam state m, v (double, length ppo_trained_count; the
 * caller zeroes them before the first step) with step counter *t.
 * stats_out (optional) receives per step: the four loss statistics of
 * ppo_loss_grad and the gradient norm before clipping.
 */
int ppo_update(float *w, const ppo_shape *s, const ppo_hp *hp, const float *states, const int32_t *actions,
               const float *logp_old, const float *adv, const float *ret, const int32_t *rows, int n_steps,
               int B, double *m, double *v, long *t, double *stats_out)
{
    const long np = ppo_trained_count(s);
    double *p = (double *)malloc(sizeof(double) * np), *g = (double *)malloc(sizeof(double) * np);
    if (!p || !g) {
        free(p);
        free(g);
        return -1;
    }
    for (long i = 0; i < np; ++i) p[i] = (double)w[i];
    for (int k = 0; k < n_steps; ++k) {
        double st[4];
        ppo_loss_grad(p, s, hp, states, actions, logp_old, adv, ret, rows + (long)k * B, B, g, st);
        *t += 1;
        const double norm = ppo_adam_step(p, g, m, v, np, *t, hp);
        if (stats_out) {
            for (int j = 0; j < 4; ++j) stats_out[k * 5 + j] = st[j];
            stats_out[k * 5 + 4] = norm;
        }
    }
    for (long i = 0; i < np; ++i) w[i] = (float)p[i];
    free(p);
    free(g);
    return 0;
}
