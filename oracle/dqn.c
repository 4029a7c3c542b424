/*
 * dqn.c -- plain, slow, single-threaded CPU statement of DQN experience
 * collection: the environment of the PPO collector (oracle.c, included here,
 * so that both collectors' oracles share one statement of the environment),
 * with a dueling Q network choosing each action epsilon-greedily and a target
 * network giving each transition its TD error.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the tests and the smoke check do.  It shares no code, header, table or
 * constant with the CUDA path.
 *
 * Sources (page titles; sections named):
 *  [P2] "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA Experience Collection":
 *       "Data Flow" (per step: features, portfolio features, online Q
 *       forward, epsilon-greedy selection with the LCG, portfolio, barrier,
 *       diversity, curiosity, next state, target Q forward, TD error, reward,
 *       store, reset on done); "Kernel Components" 1 (dueling Q network:
 *       54 -> 256 LeakyReLU(0.01) -> 256 LeakyReLU(0.01), value stream
 *       256 -> 128 LeakyReLU -> 1, advantage stream 256 -> 128 LeakyReLU -> 45,
 *       Q(s,a) = V(s) + (A(s,a) - mean_a A(s,a)); weights [out, in]),
 *       7 (TD error |r + gamma max_a' Q_target(s', a') (1 - done) -
 *       Q_online(s, a)|), 8 (the LCG); "Epsilon Decay" (epsilon a scalar per
 *       launch).
 * Readings where the page leaves a step open (each stated in the design
 * notes): the environment, curiosity and reward are the PPO collector's (the
 * workload specification's), so both collectors step the same environment;
 * each step draws two LCG uniforms: u1 decides exploration (u1 < epsilon),
 * the second state s2 gives the random action ((s2 >> 8) * n_actions) >> 24
 * (floor(u2 * n_actions), exact in integers); the greedy action is the first
 * index of the largest Q; the target network sees the pre-reset next state
 * (the curiosity target); the stored Q is the online Q of the action taken.
 * Episode recycling ("Future Phase 3 Optimization": when an episode ends,
 * start a new one from a new random bar instead of idling), an option: after
 * a done at step t < L - 1 the LCG is stepped once more and step t + 1 starts
 * at bar ((s >> 8) * R) >> 24, R = n_bars - L + t + 1 (every bar that leaves
 * room for the remaining steps and their next bars), with the portfolio reset
 * as on every done; the finished transition's next state stays the
 * pre-reset state at the bar after its own.  Without the option the episode
 * goes on at the next bar, as in the PPO collector.
 *
 * Weights: one float32 buffer [online net | target net | curiosity block],
 * each net W1 [256 x 54], b1, W2 [256 x 256], b2, Wv1 [128 x 256], bv1,
 * Wv2 [1 x 128], bv2, Wa1 [128 x 256], ba1, Wa2 [45 x 128], ba2; the
 * curiosity block as in the PPO buffer.  Mode Q as in oracle.c.
 */
#include "oracle.c"

#define DQN_H 256
#define DQN_S 128

typedef struct {
    long w1, b1, w2, b2, wv1, bv1, wv2, bv2, wa1, ba1, wa2, ba2, total;
} dqn_layout;

static void dqn_make_layout(int sd, int na, dqn_layout *lo)
{
    long off = 0;
    lo->w1 = off; off += (long)DQN_H * sd;
    lo->b1 = off; off += DQN_H;
    lo->w2 = off; off += (long)DQN_H * DQN_H;
    lo->b2 = off; off += DQN_H;
    lo->wv1 = off; off += (long)DQN_S * DQN_H;
    lo->bv1 = off; off += DQN_S;
    lo->wv2 = off; off += DQN_S;
    lo->bv2 = off; off += 1;
    lo->wa1 = off; off += (long)DQN_S * DQN_H;
    lo->ba1 = off; off += DQN_S;
    lo->wa2 = off; off += (long)na * DQN_S;
    lo->ba2 = off; off += na;
    lo->total = off;
}

long dqn_net_count(const oracle_cfg *c)
{
    dqn_layout lo;
    dqn_make_layout(c->n_market + 3, c->n_actions, &lo);
    return lo.total;
}

static void leaky(double *v, int n)
{
    for (int i = 0; i < n; ++i)
        if (v[i] < 0.0) v[i] *= 0.01;
}

/* [P2] component 1: V and the advantages A of state x under one net */
void dqn_q_parts(const float *net, const oracle_cfg *c, const double *x, double *v, double *adv)
{
    dqn_layout lo;
    const int sd = c->n_market + 3, na = c->n_actions;
    double in[ORACLE_MAX_W], h[ORACLE_MAX_W], hv[ORACLE_MAX_W], ha[ORACLE_MAX_W];
    dqn_make_layout(sd, na, &lo);
    q_vector(x, in, sd, c->quant);
    oracle_dense(net + lo.w1, net + lo.b1, DQN_H, sd, in, h, 0, c->quant);
    leaky(h, DQN_H);
    q_vector(h, in, DQN_H, c->quant);
    oracle_dense(net + lo.w2, net + lo.b2, DQN_H, DQN_H, in, h, 0, c->quant);
    leaky(h, DQN_H);
    q_vector(h, in, DQN_H, c->quant);                      /* the shared output feeds both streams */
    oracle_dense(net + lo.wv1, net + lo.bv1, DQN_S, DQN_H, in, hv, 0, c->quant);
    leaky(hv, DQN_S);
    oracle_dense(net + lo.wa1, net + lo.ba1, DQN_S, DQN_H, in, ha, 0, c->quant);
    leaky(ha, DQN_S);
    q_vector(hv, in, DQN_S, c->quant);
    oracle_dense(net + lo.wv2, net + lo.bv2, 1, DQN_S, in, v, 0, c->quant);
    q_vector(ha, in, DQN_S, c->quant);
    oracle_dense(net + lo.wa2, net + lo.ba2, na, DQN_S, in, adv, 0, c->quant);
}

/* Q(s, a) = V(s) + (A(s, a) - mean_a A(s, a)) */
void dqn_q(const float *net, const oracle_cfg *c, const double *x, double *q)
{
    double v, adv[ORACLE_MAX_W];
    const int na = c->n_actions;
    dqn_q_parts(net, c, x, &v, adv);
    double mean = 0.0;
    for (int a = 0; a < na; ++a) mean += adv[a];
    mean /= (double)na;
    for (int a = 0; a < na; ++a) q[a] = v + (adv[a] - mean);
}

static int first_argmax(const double *q, int n)
{
    int best = 0;
    for (int a = 1; a < n; ++a)
        if (q[a] > q[best]) best = a;
    return best;
}

/*
 * Episode n from bar `start`, LCG state `seed`, L steps, exploration rate
 * epsilon.  gpu_a / gpu_d (length L, may be NULL): decisions of the path under
 * test.  Where the greedy action differs from gpu_a and the gap between the
 * two actions' Q values is below q_band * max(1, max|Q|), the GPU's action is
 * adopted and counted as a replay (a floating-point decision between
 * near-equal values); any other difference is a mismatch (also adopted, so
 * that the rest of the episode can be compared).  Dones as in oracle_episode.
 * Outputs (length L, or L * state_dim) may be NULL: states, actions, rewards,
 * dones, q (online Q of the action taken), td, next_states (pre-reset), bars
 * (the bar each step's state was read from).  recycle: the option above.
 */
int dqn_episode(const float *w, const oracle_cfg *c, const float *features, long n_bars, int start,
                uint32_t seed, int L, double gamma, double epsilon, int recycle, const int32_t *gpu_a,
                const int32_t *gpu_d, double q_band, double done_band, float *o_states, int32_t *o_a, float *o_r,
                int32_t *o_d, float *o_q, float *o_td, float *o_next, int32_t *o_bars, oracle_stats *st)
{
    const int nm = c->n_market, sd = nm + 3, na = c->n_actions;
    if (L <= 0 || start < 0 || (long)start + L > n_bars - 1 || na > ORACLE_MAX_W ||
        c->div_window > ORACLE_MAX_WIN || c->div_window <= 0)
        return -1;
    const long net = dqn_net_count(c);
    const float *online = w, *target = w + net, *cw = w + 2 * net;
    double x[ORACLE_MAX_W], xn[ORACLE_MAX_W], q[ORACLE_MAX_W], qt[ORACLE_MAX_W];
    env_state es;
    env_reset(&es);
    uint32_t s = seed;
    long bar = start;

    for (int t = 0; t < L; ++t) {
        const long b = bar;
        for (int j = 0; j < nm; ++j) x[j] = (double)features[b * nm + j];
        x[nm] = es.V; x[nm + 1] = es.e; x[nm + 2] = c->spread;

        /* online Q, epsilon-greedy */
        dqn_q(online, c, x, q);
        double u1 = oracle_lcg_uniform(&s);
        s = oracle_lcg_step(s);
        int a_rand = (int)((((uint64_t)(s >> 8)) * (uint64_t)na) >> 24);
        int explore = u1 < epsilon;
        int a = explore ? a_rand : first_argmax(q, na);
        if (gpu_a && gpu_a[t] != a) {
            int g = gpu_a[t];
            double gap = INFINITY;
            if (!explore && g >= 0 && g < na) {
                double scale = 1.0;
                for (int j = 0; j < na; ++j) scale = fmax(scale, fabs(q[j]));
                gap = (q[a] - q[g]) / scale;
            }
            if (gap < q_band) st->action_replays++;
            else {
                st->action_mismatches++;
                if (gap > st->max_action_gap) st->max_action_gap = gap;
            }
            if (g >= 0 && g < na) a = g;
        }
        double q_sel = q[a];

        /* environment, curiosity, reward; xn = pre-reset next state */
        int done;
        double rew = env_step(cw, c, features, b, x, a, gpu_d ? gpu_d[t] : -1, done_band, &es, st, xn, &done,
                              NULL, NULL, NULL);

        /* target network on the next state, TD error */
        dqn_q(target, c, xn, qt);
        double mt = qt[first_argmax(qt, na)];
        double td = fabs(rew + gamma * mt * (1.0 - (double)done) - q_sel);

        if (o_states) for (int j = 0; j < sd; ++j) o_states[(long)t * sd + j] = (float)x[j];
        if (o_next) for (int j = 0; j < sd; ++j) o_next[(long)t * sd + j] = (float)xn[j];
        if (o_a) o_a[t] = a;
        if (o_r) o_r[t] = (float)rew;
        if (o_d) o_d[t] = done;
        if (o_q) o_q[t] = (float)q_sel;
        if (o_td) o_td[t] = (float)td;
        if (o_bars) o_bars[t] = (int32_t)b;

        /* the next step's bar: the next one, or after a done with recycling a
           fresh bar from the episode's LCG */
        if (recycle && done && t < L - 1) {
            s = oracle_lcg_step(s);
            const uint64_t range = (uint64_t)(n_bars - L + t + 1);
            bar = (long)((((uint64_t)(s >> 8)) * range) >> 24);
        } else {
            bar = b + 1;
        }
    }
    return 0;
}

/* episodes idx[0..n_sel-1]; per-episode outputs at row i; gpu_a / gpu_d are [N, L] */
int dqn_rollout(const float *w, const oracle_cfg *c, const float *features, long n_bars, const int32_t *starts,
                const uint32_t *seeds, const int32_t *idx, int n_sel, int L, double gamma, double epsilon,
                int recycle, const int32_t *gpu_a, const int32_t *gpu_d, double q_band, double done_band,
                float *o_states, int32_t *o_a, float *o_r, int32_t *o_d, float *o_q, float *o_td, float *o_next,
                int32_t *o_bars, oracle_stats *st)
{
    const int sd = c->n_market + 3;
    for (int i = 0; i < n_sel; ++i) {
        long n = idx[i], row = (long)i * L;
        int rc = dqn_episode(w, c, features, n_bars, starts[n], seeds[n], L, gamma, epsilon, recycle,
                             gpu_a ? gpu_a + n * L : NULL, gpu_d ? gpu_d + n * L : NULL, q_band, done_band,
                             o_states ? o_states + row * sd : NULL, o_a ? o_a + row : NULL,
                             o_r ? o_r + row : NULL, o_d ? o_d + row : NULL, o_q ? o_q + row : NULL,
                             o_td ? o_td + row : NULL, o_next ? o_next + row * sd : NULL,
                             o_bars ? o_bars + row : NULL, st);
        if (rc) return rc;
    }
    return 0;
}
