/*
 * oracle.c -- plain, slow, single-threaded CPU statement of fused PPO
 * experience collection (actor -> categorical sample -> critic -> portfolio,
 * triple-barrier, diversity and curiosity reward -> reset on done, then a
 * backward GAE scan per episode).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * path: it reads the same packed float32 weights and the same seeded inputs
 * and computes everything again from the definitions below, accumulating in
 * double.
 *
 * Sources (page titles; sections named):
 *  [P1] "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection":
 *       "Kernel Phases" (Phase A steps 1-12, Phase B GAE), "Weight Layout",
 *       "Output Buffers".
 *  [P2] "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA Experience Collection":
 *       "Kernel Components" 2 (action category for curiosity / diversity),
 *       4 (barrier labels -1/0/+1), 5 (Shannon entropy over 3 categories,
 *       log2, penalty when H < 1.0), 6 (reward = pnl*(1+barrier_scale) +
 *       diversity + curiosity - risk; barrier_scale +0.5 profit, -0.5 stop),
 *       8 (LCG s = s*1664525 + 1013904223), and the dense-layer convention
 *       out[j] = b[j] + sum_i in[i] * W[j*in + i].
 * The workload specification fixes what the pages leave open: exposure
 * {-1,-.5,0,.5,1}[a/9], cost (1+(a%9)/3+a%3)*1e-4, barriers +-theta on PnL or
 * K bars, diversity window 20 and penalty -0.01, curiosity (54+45 one-hot)->
 * 64->54 with bonus 0.01*MSE, risk 1e-3*|exposure|, uniform (s>>8)*2^-24,
 * bootstrap V_boot = critic(final pre-reset next state).
 *
 * Readings where the pages are silent (each is listed with its reason in the
 * design notes): state = [F[b,0..50], V, e, spread] with V the portfolio value
 * since the last reset (reset capital 1), e the exposure held entering the
 * step and spread the constant tx_base; the price ratio P[b+1]/P[b] is
 * exp(F[b+1,0]); V' = V*(1-|e'-e|*rate)*(1+e'*(g-1)); the barrier tests
 * V'-1 against +-theta (price barrier wins over time for the label); the
 * diversity window covers the actions since the last reset (at most 20,
 * including the current one); the curiosity target is the full pre-reset next
 * state; log p is the log-softmax (l_a - m) - ln(sum exp(l - m)); the CDF is
 * summed in index order and a = min{i : u < cdf_i}, else the last action.
 *
 * "Mode Q" (quant = 1 bf16 round-to-nearest-even, quant = 2 tf32
 * round-to-nearest-ties-away) states what a reduced-precision tensor-core path
 * computes: every weight matrix element and every layer input is rounded to
 * the operand format once, products and sums are exact (here: double), biases
 * and activations stay at full precision.  quant = 0 rounds nothing.
 *
 * Rounding replay (mode Q only).  A tensor-core path accumulates each hidden
 * pre-activation z in float32 before rounding it to the operand format, so
 * where the exact z lies within float32 accumulation error of a rounding
 * boundary (the midpoint between two neighbouring bf16 / tf32 values, or 0
 * for the ReLU) the path may round to the other neighbour.  That is a
 * floating-point decision like an action drawn within rounding of a CDF
 * boundary, and it is handled the same way: given the path's rounded hidden
 * activations, the oracle adopts the path's value where it is the rounding
 * of some point within the bound of the exact z (a replay), and counts any
 * other difference as a mismatch (adopted as well, so that the rest can still
 * be compared).  The bound for a K-term sum of products plus bias, whose
 * magnitudes sum to S, is (K + 4) * 2^-23 * S: the standard error bound of
 * recursive float32 summation (Higham, "Accuracy and Stability of Numerical
 * Algorithms", section 4.2), charged a whole unit in the last place per
 * operation so that accumulators that truncate are covered, with four
 * operations to spare for bias and epilogue additions.  The state input is
 * rounded the same way from the path's own float32 state, whose portfolio
 * value may differ from the oracle's double one within the state tolerance
 * (state_band, relative to max(|x|, 1)); its rounding is replayed within that
 * band.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_W 1024   /* widest layer supported */
#define ORACLE_MAX_WIN 256  /* longest diversity window supported */

typedef struct {
    int n_market;        /* market features per bar (51) */
    int n_actions;       /* actions (45) */
    int actor_h1;        /* 128 */
    int actor_h2;        /* 64 */
    int critic_nh;       /* hidden layers of the critic (5) */
    int critic_h[8];     /* their widths */
    int cur_h;           /* curiosity hidden width (64) */
    int quant;           /* 0 none, 1 bf16 RNE, 2 tf32 RNA */
    double barrier;      /* theta */
    int max_hold;        /* K */
    double pt_scale;     /* barrier_scale on a profit-take hit */
    double sl_scale;     /* barrier_scale on a stop-loss hit */
    int div_window;      /* 20 */
    double div_thresh;   /* 1.0 */
    double div_penalty;  /* -0.01 */
    double cur_coef;     /* 0.01 */
    double risk_coef;    /* 1e-3 */
    double tx_base;      /* 1e-4 */
    double spread;       /* portfolio feature 3 (constant) */
} oracle_cfg;

typedef struct {
    long action_replays;     /* GPU action adopted: oracle differed inside the band */
    long done_replays;       /* GPU done adopted: oracle differed inside the band */
    long action_mismatches;  /* differed outside the band */
    long done_mismatches;
    double max_action_gap;   /* largest |u - cdf boundary| among action differences */
    double max_done_gap;     /* largest |V'-1 -+ theta| among done differences */
    long hidden_replays;     /* hidden roundings adopted from the path under test (inside the bound) */
    long hidden_mismatches;  /* hidden values of the path that no point within the bound rounds to */
    double max_hidden_excess;/* largest distance of such a value from the allowed interval, in bounds */
} oracle_stats;

/* ------------------------------------------------------------------ */
/* LCG ([P2] "Epsilon-Greedy RNG"; uniform from the top 24 state bits)  */
/* ------------------------------------------------------------------ */

uint32_t oracle_lcg_step(uint32_t s)
{
    return (uint32_t)((uint64_t)s * 1664525u + 1013904223u); /* mod 2^32 */
}

/* advances *s once and returns u = (s >> 8) * 2^-24 in [0, 1) */
double oracle_lcg_uniform(uint32_t *s)
{
    *s = oracle_lcg_step(*s);
    return (double)(*s >> 8) / 16777216.0;
}

/* n consecutive uniforms from state seed */
void oracle_lcg_fill(uint32_t seed, long n, double *out)
{
    uint32_t s = seed;
    for (long i = 0; i < n; ++i) out[i] = oracle_lcg_uniform(&s);
}

/* ------------------------------------------------------------------ */
/* operand rounding for mode Q                                          */
/* ------------------------------------------------------------------ */

static uint32_t f2u(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float u2f(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* IEEE round-to-nearest-even of a float to 8 significant bits (bfloat16). */
float oracle_round_bf16(float x)
{
    uint32_t u = f2u(x);
    if ((u & 0x7f800000u) == 0x7f800000u) return x;          /* inf / nan */
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return u2f(u & 0xffff0000u);
}

/* round-to-nearest, ties away from zero, to 11 significant bits (tf32). */
float oracle_round_tf32(float x)
{
    uint32_t u = f2u(x);
    if ((u & 0x7f800000u) == 0x7f800000u) return x;
    u += 0x1000u;                 /* half an ulp of the 10-bit mantissa */
    return u2f(u & 0xffffe000u);
}

static double q_operand(double v, int quant)
{
    if (quant == 0) return v;
    float f = (float)v;
    return (double)(quant == 1 ? oracle_round_bf16(f) : oracle_round_tf32(f));
}

/* ------------------------------------------------------------------ */
/* dense layers ([P2] "Kernel Components" 1, weight layout [out, in])   */
/* ------------------------------------------------------------------ */

/* out[j] = b[j] + sum_i W[j*n_in + i] * in[i], optional ReLU.
 * Under mode Q the weights are rounded here and the caller passes an input
 * vector that has already been rounded. */
void oracle_dense(const float *W, const float *b, int n_out, int n_in,
                  const double *in, double *out, int relu, int quant)
{
    for (int j = 0; j < n_out; ++j) {
        double acc = 0.0;
        for (int i = 0; i < n_in; ++i)
            acc += q_operand((double)W[(long)j * n_in + i], quant) * in[i];
        acc += (double)b[j];
        out[j] = (relu && acc < 0.0) ? 0.0 : acc;
    }
}

/* The float32 accumulation bound of a K-term dot product plus bias whose
 * terms' magnitudes sum to S (see "Rounding replay" above). */
static double accum_bound(int K, double S) { return (double)(K + 4) * ldexp(S, -23); }

/* oracle_dense followed by the operand rounding of the next layer's input
 * (relu and quant as oracle_dense / q_operand).  gpu (may be NULL): the path
 * under test's rounded outputs for the same layer; where they differ from the
 * oracle's, they are adopted as described under "Rounding replay". */
static void dense_round_replay(const float *W, const float *b, int n_out, int n_in, const double *in,
                               double *out, int relu, int quant, const float *gpu, oracle_stats *st)
{
    for (int j = 0; j < n_out; ++j) {
        double acc = 0.0, mag = fabs((double)b[j]);
        for (int i = 0; i < n_in; ++i) {
            double p = q_operand((double)W[(long)j * n_in + i], quant) * in[i];
            acc += p;
            mag += fabs(p);
        }
        acc += (double)b[j];
        double own = q_operand((relu && acc < 0.0) ? 0.0 : acc, quant);
        out[j] = own;
        if (!gpu || (double)gpu[j] == own) continue;
        double g = (double)gpu[j], d = accum_bound(n_in, mag);
        double zl = acc - d, zh = acc + d;
        if (relu) { zl = zl < 0.0 ? 0.0 : zl; zh = zh < 0.0 ? 0.0 : zh; }
        double lo = q_operand(zl, quant), hi = q_operand(zh, quant);
        if (g >= lo && g <= hi) {
            st->hidden_replays++;
        } else {
            double ex = (g < lo ? lo - g : g - hi) / (d > 0.0 ? d : 1.0);
            st->hidden_mismatches++;
            if (ex > st->max_hidden_excess || !(ex == ex)) st->max_hidden_excess = ex;
        }
        out[j] = g;
    }
}

/* The operand rounding of a state input x[0..n) into xq, given the path's
 * rounded input gpu (may be NULL): a different value is adopted as a replay
 * when it is the rounding of a point within band * max(|x_j|, 1) of x_j, and
 * as a mismatch otherwise. */
static void input_round_replay(const double *x, int n, int quant, const float *gpu, double band, double *xq,
                               oracle_stats *st)
{
    for (int j = 0; j < n; ++j) {
        double own = q_operand(x[j], quant);
        xq[j] = own;
        if (!gpu || (double)gpu[j] == own) continue;
        double g = (double)gpu[j], d = band * fmax(fabs(x[j]), 1.0);
        double lo = q_operand(x[j] - d, quant), hi = q_operand(x[j] + d, quant);
        if (g >= lo && g <= hi) {
            st->hidden_replays++;
        } else {
            double ex = (g < lo ? lo - g : g - hi) / (d > 0.0 ? d : 1.0);
            st->hidden_mismatches++;
            if (ex > st->max_hidden_excess || !(ex == ex)) st->max_hidden_excess = ex;
        }
        xq[j] = g;
    }
}

/* dense_round_replay for the pins: one layer's rounded outputs `out`, given
 * the path's rounded outputs `gpu` (may be NULL); counts in *st */
void oracle_dense_round_replay(const float *W, const float *b, int n_out, int n_in, const double *in,
                               double *out, int relu, int quant, const float *gpu, oracle_stats *st)
{
    dense_round_replay(W, b, n_out, n_in, in, out, relu, quant, gpu, st);
}

static void q_vector(const double *in, double *out, int n, int quant)
{
    for (int i = 0; i < n; ++i) out[i] = q_operand(in[i], quant);
}

/* offsets into the packed weight buffer ([P1] "Weight Layout" order:
 * actor, critic, curiosity; each matrix followed by its bias) */
typedef struct {
    long a_w[3], a_b[3];
    long c_w[9], c_b[9];
    long q_w[2], q_b[2];
    int a_in[3], a_out[3];
    int c_in[9], c_out[9];
    int q_in[2], q_out[2];
    int n_critic;          /* layers including the scalar head */
} layout;

static void make_layout(const oracle_cfg *c, layout *lo)
{
    long off = 0;
    int sd = c->n_market + 3;
    int ain[3] = {sd, c->actor_h1, c->actor_h2};
    int aout[3] = {c->actor_h1, c->actor_h2, c->n_actions};
    for (int l = 0; l < 3; ++l) {
        lo->a_in[l] = ain[l]; lo->a_out[l] = aout[l];
        lo->a_w[l] = off; off += (long)ain[l] * aout[l];
        lo->a_b[l] = off; off += aout[l];
    }
    int prev = sd;
    lo->n_critic = c->critic_nh + 1;
    for (int l = 0; l < lo->n_critic; ++l) {
        int o = (l < c->critic_nh) ? c->critic_h[l] : 1;
        lo->c_in[l] = prev; lo->c_out[l] = o;
        lo->c_w[l] = off; off += (long)prev * o;
        lo->c_b[l] = off; off += o;
        prev = o;
    }
    int qin[2] = {sd + c->n_actions, c->cur_h};
    int qout[2] = {c->cur_h, sd};
    for (int l = 0; l < 2; ++l) {
        lo->q_in[l] = qin[l]; lo->q_out[l] = qout[l];
        lo->q_w[l] = off; off += (long)qin[l] * qout[l];
        lo->q_b[l] = off; off += qout[l];
    }
}

long oracle_weight_count(const oracle_cfg *c)
{
    layout lo;
    make_layout(c, &lo);
    return lo.q_b[1] + lo.q_out[1];
}

/* [P1] Phase A step 3: state[54] -> h1[128] ReLU -> h2[64] ReLU -> logits[45].
 * gpu_h (may be NULL): the path's rounded h1 | h2, replayed (mode Q).
 * used_h (may be NULL) receives the h1 | h2 the logits were computed from.
 * xq (may be NULL): the already rounded state input. */
static void actor_replay(const float *w, const oracle_cfg *c, const double *x, double *logits,
                         const float *gpu_h, oracle_stats *st, float *used_h, const double *xq)
{
    long at = 0;
    layout lo;
    double in[ORACLE_MAX_W], out[ORACLE_MAX_W];
    make_layout(c, &lo);
    if (xq) memcpy(in, xq, sizeof(double) * (size_t)lo.a_in[0]);
    else q_vector(x, in, lo.a_in[0], c->quant);
    for (int l = 0; l < 3; ++l) {
        if (l == 2) {
            oracle_dense(w + lo.a_w[l], w + lo.a_b[l], lo.a_out[l], lo.a_in[l], in, logits, 0, c->quant);
        } else {
            if (gpu_h && c->quant) {
                dense_round_replay(w + lo.a_w[l], w + lo.a_b[l], lo.a_out[l], lo.a_in[l], in, out, 1, c->quant,
                                   gpu_h + at, st);
                memcpy(in, out, sizeof(double) * (size_t)lo.a_out[l]);
            } else {
                oracle_dense(w + lo.a_w[l], w + lo.a_b[l], lo.a_out[l], lo.a_in[l], in, out, 1, c->quant);
                q_vector(out, in, lo.a_out[l], c->quant);
            }
            if (used_h) for (int j = 0; j < lo.a_out[l]; ++j) used_h[at + j] = (float)in[j];
            at += lo.a_out[l];
        }
    }
}

void oracle_actor(const float *w, const oracle_cfg *c, const double *x, double *logits)
{
    actor_replay(w, c, x, logits, NULL, NULL, NULL, NULL);
}

/* [P1] Phase A step 5: state[54] -> 512 -> 384 -> 256 -> 128 -> 64 (ReLU) -> 1.
 * gpu_h (may be NULL): the path's rounded hidden layers, concatenated, replayed (mode Q).
 * used_h (may be NULL) receives the hidden layers the value was computed from.
 * xq (may be NULL): the already rounded state input. */
static double critic_replay(const float *w, const oracle_cfg *c, const double *x, const float *gpu_h,
                            oracle_stats *st, float *used_h, const double *xq)
{
    layout lo;
    double in[ORACLE_MAX_W], out[ORACLE_MAX_W];
    make_layout(c, &lo);
    if (xq) memcpy(in, xq, sizeof(double) * (size_t)lo.c_in[0]);
    else q_vector(x, in, lo.c_in[0], c->quant);
    long at = 0;
    for (int l = 0; l < lo.n_critic; ++l) {
        int last = (l == lo.n_critic - 1);
        if (last) {
            oracle_dense(w + lo.c_w[l], w + lo.c_b[l], lo.c_out[l], lo.c_in[l], in, out, 0, c->quant);
            return out[0];
        }
        if (gpu_h && c->quant) {
            dense_round_replay(w + lo.c_w[l], w + lo.c_b[l], lo.c_out[l], lo.c_in[l], in, out, 1, c->quant,
                               gpu_h + at, st);
            memcpy(in, out, sizeof(double) * (size_t)lo.c_out[l]);
        } else {
            oracle_dense(w + lo.c_w[l], w + lo.c_b[l], lo.c_out[l], lo.c_in[l], in, out, 1, c->quant);
            q_vector(out, in, lo.c_out[l], c->quant);
        }
        if (used_h) for (int j = 0; j < lo.c_out[l]; ++j) used_h[at + j] = (float)in[j];
        at += lo.c_out[l];
    }
    return 0.0;
}

double oracle_critic(const float *w, const oracle_cfg *c, const double *x)
{
    return critic_replay(w, c, x, NULL, NULL, NULL, NULL);
}

/* [P1] Phase A step 9 / [P2] "Curiosity Forward Model": forward-dynamics
 * prediction from [state ; one-hot(action)] -> cur_h ReLU -> next state.
 * cw points at the curiosity block [C1 (cur_h x (sd + n_actions)), c1,
 * C2 (sd x cur_h), c2]. */
static void curiosity_block(const float *cw, const oracle_cfg *c, const double *x, int a, double *pred,
                            const float *gpu_z, oracle_stats *st, float *used_z, const double *xq)
{
    double in[ORACLE_MAX_W], hid[ORACLE_MAX_W];
    const int sd = c->n_market + 3, nin = sd + c->n_actions, h = c->cur_h;
    const float *C1 = cw, *c1 = C1 + (long)h * nin, *C2 = c1 + h, *c2 = C2 + (long)sd * h;
    if (xq) memcpy(in, xq, sizeof(double) * (size_t)sd);
    else q_vector(x, in, sd, c->quant);
    for (int i = 0; i < c->n_actions; ++i) in[sd + i] = (i == a) ? 1.0 : 0.0;
    if (gpu_z && c->quant) {
        dense_round_replay(C1, c1, h, nin, in, hid, 1, c->quant, gpu_z, st);
        memcpy(in, hid, sizeof(double) * (size_t)h);
    } else {
        oracle_dense(C1, c1, h, nin, in, hid, 1, c->quant);
        q_vector(hid, in, h, c->quant);
    }
    if (used_z) for (int j = 0; j < h; ++j) used_z[j] = (float)in[j];
    oracle_dense(C2, c2, sd, h, in, pred, 0, c->quant);
}

void oracle_curiosity(const float *w, const oracle_cfg *c, const double *x, int a, double *pred)
{
    layout lo;
    make_layout(c, &lo);
    curiosity_block(w + lo.q_w[0], c, x, a, pred, NULL, NULL, NULL, NULL);
}

/* Columns of one row of the path's rounded operands (see oracle_episode):
 * state input (ORACLE_IN_COLS, the first n_market + 3 used) | actor h1 |
 * actor h2 | critic hidden layers | curiosity hidden. */
#define ORACLE_IN_COLS 64
long oracle_hidden_width(const oracle_cfg *c)
{
    long wd = ORACLE_IN_COLS + c->actor_h1 + c->actor_h2 + c->cur_h;
    for (int l = 0; l < c->critic_nh; ++l) wd += c->critic_h[l];
    return wd;
}

/* [P1] Phase A step 4: stable softmax, CDF summed in index order, inverse-CDF
 * draw with uniform u.  Returns the action; writes log p[action] and the CDF. */
int oracle_sample(const double *logits, int n, double u, double *logp, double *cdf)
{
    double m = logits[0];
    for (int i = 1; i < n; ++i) if (logits[i] > m) m = logits[i];
    double q[ORACLE_MAX_W], s = 0.0;
    for (int i = 0; i < n; ++i) { q[i] = exp(logits[i] - m); s += q[i]; }
    double run = 0.0;
    int a = -1;
    for (int i = 0; i < n; ++i) {
        run += q[i] / s;
        cdf[i] = run;
        if (a < 0 && u < run) a = i;
    }
    if (a < 0) a = n - 1;
    *logp = (logits[a] - m) - log(s);
    return a;
}

/* log p[a] for a given action (used when the GPU's action is adopted). */
static double log_prob(const double *logits, int n, int a)
{
    double m = logits[0];
    for (int i = 1; i < n; ++i) if (logits[i] > m) m = logits[i];
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += exp(logits[i] - m);
    return (logits[a] - m) - log(s);
}

/* ------------------------------------------------------------------ */
/* environment ([P1] steps 6-10, [P2] components 3-6)                   */
/* ------------------------------------------------------------------ */

double oracle_exposure(int a) { return 0.5 * (double)(a / 9 - 2); } /* {-1,-.5,0,.5,1} */

double oracle_tx_rate(int a, double base) { return (double)(1 + (a % 9) / 3 + a % 3) * base; }

/* [P2] component 2: Short (exposure index 0,1) / Flat (2) / Long (3,4) */
int oracle_category(int a)
{
    int x = a / 9;
    return (x <= 1) ? 0 : (x == 2) ? 1 : 2;
}

/* [P2] component 5: Shannon entropy (bits) of the category histogram */
double oracle_window_entropy(const int *cats, int n)
{
    if (n <= 0) return 0.0;
    int cnt[3] = {0, 0, 0};
    for (int i = 0; i < n; ++i) cnt[cats[i]]++;
    double h = 0.0;
    for (int k = 0; k < 3; ++k) {
        if (cnt[k] == 0) continue;
        double p = (double)cnt[k] / (double)n;
        h -= p * log2(p);
    }
    return h;
}

/* [P1] Phase B: backward GAE over one episode.  v_boot is V(next) of the last
 * step; (1 - d) masks the bootstrap and the recursion at episode ends. */
void oracle_gae(const double *r, const double *v, const int32_t *d, int L, double v_boot,
                double gamma, double lambda, double *adv, double *ret)
{
    double next_adv = 0.0;
    for (int t = L - 1; t >= 0; --t) {
        double v_next = (t == L - 1) ? v_boot : v[t + 1];
        double nd = d[t] ? 0.0 : 1.0;
        double delta = r[t] + gamma * v_next * nd - v[t];
        adv[t] = delta + gamma * lambda * nd * next_adv;
        next_adv = adv[t];
        ret[t] = adv[t] + v[t];
    }
}

/* float entry point for the GAE pins */
void oracle_gae_f32(const float *r, const float *v, const int32_t *d, int L, double v_boot,
                    double gamma, double lambda, double *adv, double *ret)
{
    double *rr = malloc(sizeof(double) * (size_t)L), *vv = malloc(sizeof(double) * (size_t)L);
    for (int t = 0; t < L; ++t) { rr[t] = r[t]; vv[t] = v[t]; }
    oracle_gae(rr, vv, d, L, v_boot, gamma, lambda, adv, ret);
    free(rr); free(vv);
}

/* ------------------------------------------------------------------ */
/* one environment step ([P1] steps 6-10)                               */
/* ------------------------------------------------------------------ */

typedef struct {
    double V, e;                 /* portfolio value since reset, exposure entering the step */
    int k;                       /* steps since reset */
    int nwin;                    /* actions in the diversity window */
    int win[ORACLE_MAX_WIN];     /* their categories, oldest first */
} env_state;

static void env_reset(env_state *s) { s->V = 1.0; s->e = 0.0; s->k = 0; s->nwin = 0; }

/* Portfolio, triple barrier, diversity, curiosity and reward for action a at
 * bar b, from state x (= [F[b], V, e, spread]).  Fills xn with the pre-reset
 * next state [F[b+1], V', e', spread].  gpu_done (or -1): the done decision of
 * the path under test, adopted as in oracle_episode; gpu_z (or NULL): its
 * rounded curiosity hidden layer, replayed; used_z (or NULL) receives the
 * curiosity hidden layer used; xq (or NULL): the rounded state input.  Sets *done; the state's
 * V, e, k and window advance, and are reset when *done. */
static double env_step(const float *cw, const oracle_cfg *c, const float *features, long b, const double *x,
                       int a, int gpu_done, double done_band, env_state *es, oracle_stats *st, double *xn,
                       int *done_out, const float *gpu_z, float *used_z, const double *xq)
{
    const int nm = c->n_market, sd = nm + 3;
    double pred[ORACLE_MAX_W];

    /* step 6: portfolio */
    double e2 = oracle_exposure(a);
    double rate = oracle_tx_rate(a, c->tx_base);
    double g = exp((double)features[(b + 1) * nm + 0]);
    double V2 = es->V * (1.0 - fabs(e2 - es->e) * rate) * (1.0 + e2 * (g - 1.0));
    double pnl = V2 / es->V - 1.0;

    /* step 7: triple barrier */
    es->k += 1;
    double cpl = V2 - 1.0;
    int label = (cpl >= c->barrier) ? 1 : (cpl <= -c->barrier) ? -1 : 0;
    int done = (label != 0) || (es->k >= c->max_hold);
    if (gpu_done >= 0 && (gpu_done != 0) != done) {
        double gap = fmin(fabs(cpl - c->barrier), fabs(cpl + c->barrier));
        if (gap < done_band) st->done_replays++;
        else {
            st->done_mismatches++;
            if (gap > st->max_done_gap) st->max_done_gap = gap;
        }
        done = gpu_done != 0;
        if (!done) label = 0;
        else if (es->k < c->max_hold || label == 0)
            label = (fabs(cpl - c->barrier) <= fabs(cpl + c->barrier)) ? 1 : -1;
    }

    /* step 8: diversity over the actions since reset (window of div_window) */
    if (es->nwin == c->div_window) {
        memmove(es->win, es->win + 1, sizeof(int) * (size_t)(es->nwin - 1));
        es->nwin--;
    }
    es->win[es->nwin++] = oracle_category(a);
    double H = oracle_window_entropy(es->win, es->nwin);
    double div = (H < c->div_thresh) ? c->div_penalty : 0.0;

    /* step 9: curiosity against the pre-reset next state */
    for (int j = 0; j < nm; ++j) xn[j] = (double)features[(b + 1) * nm + j];
    xn[nm] = V2; xn[nm + 1] = e2; xn[nm + 2] = c->spread;
    curiosity_block(cw, c, x, a, pred, gpu_z, st, used_z, xq);
    double mse = 0.0;
    for (int j = 0; j < sd; ++j) mse += (pred[j] - xn[j]) * (pred[j] - xn[j]);
    mse /= (double)sd;
    double cur = c->cur_coef * mse;

    /* step 10: reward */
    double risk = c->risk_coef * fabs(e2);
    double beta = (label > 0) ? c->pt_scale : (label < 0) ? c->sl_scale : 0.0;
    double rew = pnl * (1.0 + beta) + div + cur - risk;

    /* step 12: reset on done (the caller's LCG is not reseeded, the bar keeps advancing) */
    if (done) env_reset(es);
    else { es->V = V2; es->e = e2; }
    *done_out = done;
    return rew;
}

/* ------------------------------------------------------------------ */
/* one episode                                                          */
/* ------------------------------------------------------------------ */

/*
 * Runs episode n from bar `start` with LCG state `seed` for L steps.
 * features: [n_bars, n_market] float32 row-major.
 * gpu_a / gpu_d (length L, may be NULL): decisions of the path under test.
 *   Where the oracle's own action (done) differs from it and the uniform lies
 *   within act_band of the CDF boundary that separates them (|V'-1 -+ theta|
 *   < done_band), the oracle adopts it and counts a replay.  A difference
 *   outside the band is counted as a mismatch and also adopted, so that the
 *   rest of the episode can still be compared.
 * gpu_h ((L + 1) rows of oracle_hidden_width(c) floats, or NULL): the path
 *   under test's rounded operands, row t for step t (state input | actor h1 |
 *   h2 | critic hidden layers | curiosity hidden) and row L for the bootstrap
 *   critic (its state input and critic columns only); under mode Q they are
 *   replayed as described under "Rounding replay", the state input within
 *   state_band.
 * o_h ((L + 1) rows in gpu_h's layout, or NULL) receives the hidden
 *   activations the oracle used (after any replay).
 * Outputs (each of length L, or L*state_dim for states) may be NULL.
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_episode(const float *w, const oracle_cfg *c, const float *features, long n_bars,
                   int start, uint32_t seed, int L, double gamma, double lambda,
                   const int32_t *gpu_a, const int32_t *gpu_d, double act_band, double done_band,
                   const float *gpu_h, double state_band, float *o_h,
                   float *o_states, int32_t *o_a, float *o_logp, float *o_v, float *o_r,
                   int32_t *o_d, float *o_adv, float *o_ret, double *o_vboot, oracle_stats *st)
{
    const int nm = c->n_market, sd = nm + 3, na = c->n_actions;
    const long hw = oracle_hidden_width(c), h_act = ORACLE_IN_COLS, h_crit = h_act + c->actor_h1 + c->actor_h2,
               h_cur = hw - c->cur_h;
    double xq[ORACLE_MAX_W];
    if (L <= 0 || start < 0 || (long)start + L > n_bars - 1 || na > ORACLE_MAX_W ||
        c->div_window > ORACLE_MAX_WIN || c->div_window <= 0)
        return -1;

    double *r = malloc(sizeof(double) * (size_t)L), *v = malloc(sizeof(double) * (size_t)L);
    int32_t *d = malloc(sizeof(int32_t) * (size_t)L);
    double x[ORACLE_MAX_W], xn[ORACLE_MAX_W], logits[ORACLE_MAX_W], cdf[ORACLE_MAX_W];
    env_state es;
    env_reset(&es);
    uint32_t s = seed;
    layout lo;
    make_layout(c, &lo);

    for (int t = 0; t < L; ++t) {
        long b = (long)start + t;
        /* steps 1-2: market features and portfolio features */
        for (int j = 0; j < nm; ++j) x[j] = (double)features[b * nm + j];
        x[nm] = es.V; x[nm + 1] = es.e; x[nm + 2] = c->spread;

        const float *gh = (gpu_h && c->quant) ? gpu_h + (long)t * hw : NULL;
        float *oh = o_h ? o_h + (long)t * hw : NULL;
        const double *xqp = NULL;
        if (gh) {
            input_round_replay(x, sd, c->quant, gh, state_band, xq, st);
            xqp = xq;
        } else if (oh) {
            q_vector(x, xq, sd, c->quant);
        }
        if (oh) for (int j = 0; j < sd; ++j) oh[j] = (float)xq[j];

        /* steps 3-4: actor, softmax, CDF draw */
        actor_replay(w, c, x, logits, gh ? gh + h_act : NULL, st, oh ? oh + h_act : NULL, xqp);
        double u = oracle_lcg_uniform(&s);
        double logp;
        int a = oracle_sample(logits, na, u, &logp, cdf);
        if (gpu_a && gpu_a[t] != a) {
            int g = gpu_a[t];
            double gap;
            if (g < 0 || g >= na) gap = INFINITY;
            else if (g < a) gap = u - cdf[g];          /* GPU saw u below cdf[g] */
            else gap = cdf[g - 1] - u;                 /* GPU saw u at/above cdf[g-1] */
            if (gap < act_band) st->action_replays++;
            else {
                st->action_mismatches++;
                if (gap > st->max_action_gap) st->max_action_gap = gap;
            }
            if (g >= 0 && g < na) { a = g; logp = log_prob(logits, na, a); }
        }

        /* step 5: critic */
        double val = critic_replay(w, c, x, gh ? gh + h_crit : NULL, st, oh ? oh + h_crit : NULL, xqp);

        /* steps 6-10 and 12 */
        int done;
        double rew = env_step(w + lo.q_w[0], c, features, b, x, a, gpu_d ? gpu_d[t] : -1, done_band, &es, st,
                              xn, &done, gh ? gh + h_cur : NULL, oh ? oh + h_cur : NULL, xqp);

        /* step 11: store */
        if (o_states) for (int j = 0; j < sd; ++j) o_states[(long)t * sd + j] = (float)x[j];
        if (o_a) o_a[t] = a;
        if (o_logp) o_logp[t] = (float)logp;
        if (o_v) o_v[t] = (float)val;
        if (o_r) o_r[t] = (float)rew;
        if (o_d) o_d[t] = done;
        r[t] = rew; v[t] = val; d[t] = done;
    }

    /* bootstrap: critic of the final pre-reset next state */
    const float *gb = (gpu_h && c->quant) ? gpu_h + (long)L * hw : NULL;
    float *ob = o_h ? o_h + (long)L * hw : NULL;
    const double *xbp = NULL;
    if (gb) {
        input_round_replay(xn, sd, c->quant, gb, state_band, xq, st);
        xbp = xq;
    } else if (ob) {
        q_vector(xn, xq, sd, c->quant);
    }
    if (ob) for (int j = 0; j < sd; ++j) ob[j] = (float)xq[j];
    double vboot = critic_replay(w, c, xn, gb ? gb + h_crit : NULL, st, ob ? ob + h_crit : NULL, xbp);
    if (o_vboot) *o_vboot = vboot;

    double *adv = malloc(sizeof(double) * (size_t)L), *ret = malloc(sizeof(double) * (size_t)L);
    oracle_gae(r, v, d, L, vboot, gamma, lambda, adv, ret);
    for (int t = 0; t < L; ++t) {
        if (o_adv) o_adv[t] = (float)adv[t];
        if (o_ret) o_ret[t] = (float)ret[t];
    }
    free(adv); free(ret); free(r); free(v); free(d);
    return 0;
}

/*
 * Runs episodes idx[0..n_sel-1] of a batch.  Per-episode outputs are written
 * at row i of the [n_sel, L(, state_dim)] output arrays.  gpu_a / gpu_d, when
 * given, are the path-under-test's full [N, L] arrays; gpu_h (or NULL) holds
 * its hidden activations of episodes 0..n_h-1, (L + 1) rows each (see
 * oracle_episode), replayed for those episodes; o_h (or NULL) receives the
 * oracle's, (L + 1) rows per selected episode.
 */
int oracle_rollout(const float *w, const oracle_cfg *c, const float *features, long n_bars,
                   const int32_t *starts, const uint32_t *seeds, const int32_t *idx, int n_sel,
                   int L, double gamma, double lambda,
                   const int32_t *gpu_a, const int32_t *gpu_d, double act_band, double done_band,
                   const float *gpu_h, int n_h, double state_band, float *o_h,
                   float *o_states, int32_t *o_a, float *o_logp, float *o_v, float *o_r,
                   int32_t *o_d, float *o_adv, float *o_ret, double *o_vboot, oracle_stats *st)
{
    const int sd = c->n_market + 3;
    const long hw = oracle_hidden_width(c);
    for (int i = 0; i < n_sel; ++i) {
        long n = idx[i];
        long row = (long)i * L;
        int rc = oracle_episode(w, c, features, n_bars, starts[n], seeds[n], L, gamma, lambda,
                                gpu_a ? gpu_a + n * L : NULL, gpu_d ? gpu_d + n * L : NULL,
                                act_band, done_band,
                                (gpu_h && n < n_h) ? gpu_h + n * (long)(L + 1) * hw : NULL, state_band,
                                o_h ? o_h + (long)i * (L + 1) * hw : NULL,
                                o_states ? o_states + row * sd : NULL,
                                o_a ? o_a + row : NULL, o_logp ? o_logp + row : NULL,
                                o_v ? o_v + row : NULL, o_r ? o_r + row : NULL,
                                o_d ? o_d + row : NULL, o_adv ? o_adv + row : NULL,
                                o_ret ? o_ret + row : NULL, o_vboot ? o_vboot + i : NULL, st);
        if (rc) return rc;
    }
    return 0;
}
