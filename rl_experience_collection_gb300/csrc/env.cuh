// env.cuh -- per-episode environment step on the device (float32).
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A steps 4 and 6-12, with the environment
// functions of page "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA Experience
// Collection", section "Kernel Components" (3 portfolio, 4 barrier,
// 5 diversity entropy, 6 reward, 8 LCG):
//   uniform     s <- s*1664525 + 1013904223 (mod 2^32), u = (s >> 8) * 2^-24
//   action      a = min{i : u < cdf_i}, cdf summed in index order; else the last
//   exposure    e' = {-1,-.5,0,.5,1}[a/9]; cost rate (1 + (a%9)/3 + a%3) * tx_base
//   portfolio   V' = V * (1 - |e'-e| * rate) * (1 + e' * (P[b+1]/P[b] - 1)),
//               P[b+1]/P[b] = exp(F[b+1, 0]); pnl = V'/V - 1
//   barrier     k += 1; label +1 if V'-1 >= theta, -1 if <= -theta, else 0;
//               done = label != 0 or k >= K
//   diversity   Shannon entropy (bits) of the Short/Flat/Long histogram of
//               the actions since reset (last div_window); penalty if H < thr
//   reward      pnl * (1 + barrier_scale(label)) + diversity - risk * |e'|
//               (+ the curiosity bonus, added by the value phase)
//   reset       on done: V = 1, e = 0, k = 0, window cleared; the LCG and the
//               bar index keep advancing.
#pragma once

#include <stdint.h>

#include "internal.cuh"

namespace rl {

struct EpState {
    float V;          // portfolio value since the last reset (reset capital 1)
    float e;          // exposure held entering the step
    int k;            // steps since the last reset
    int nwin;         // actions in the diversity window
    uint64_t win;     // 2-bit categories, newest in bits [0,2)
    uint32_t hist;    // histogram of the window: n_short * 1024 + n_flat * 32 + n_long (each <= 31)
    uint32_t rng;     // LCG state
};

__device__ __forceinline__ void ep_reset(EpState &s)
{
    s.V = 1.0f;
    s.e = 0.0f;
    s.k = 0;
    s.nwin = 0;
    s.win = 0;
    s.hist = 0;
}

// the histogram word's unit for category c (Short 0 / Flat 1 / Long 2)
__device__ __forceinline__ uint32_t hist_unit(int c) { return 1u << (5 * (2 - c)); }

__device__ __forceinline__ float lcg_uniform(uint32_t &s)
{
    s = s * 1664525u + 1013904223u;
    return (float)(s >> 8) * (1.0f / 16777216.0f);   // exact: 24-bit integer * 2^-24
}

// Softmax + inverse-CDF draw over n logits held in a register/local array.
// Compares u * S < running sum (S = sum of exp(l - max)), i.e. u < cdf_i.
template <int N>
__device__ __forceinline__ int sample_action(const float (&l)[N], float u, float &logp)
{
    float m = l[0];
#pragma unroll
    for (int i = 1; i < N; ++i) m = fmaxf(m, l[i]);
    float q[N];
    float s = 0.0f;
#pragma unroll
    for (int i = 0; i < N; ++i) { q[i] = expf(l[i] - m); s += q[i]; }
    const float thr = u * s;
    float run = 0.0f;
    int a = N - 1;
    bool found = false;
#pragma unroll
    for (int i = 0; i < N; ++i) {
        run += q[i];
        if (!found && thr < run) { a = i; found = true; }
    }
    float la = l[0];
#pragma unroll
    for (int i = 1; i < N; ++i) la = (i == a) ? l[i] : la;
    logp = (la - m) - logf(s);
    return a;
}

// The portfolio part of a step for action a, given em1 = expm1(F[b+1, 0]) (the
// bar's simple return): trade cost, P&L, V', the triple-barrier label and
// done.  Updates V, e and the holding time k (reset to 1, 0, 0 on done); the
// diversity window is left to env_window_reward.
__device__ __forceinline__ void env_trade(EpState &s, int a, float em1, const EnvConst &c, float &pnl,
                                          float &v_post, int &label, int &done)
{
    const int xi = a / 9;
    const float e2 = 0.5f * (float)(xi - 2);
    const float rate = (float)(1 + (a % 9) / 3 + a % 3) * c.tx_base;
    const float cost = fabsf(e2 - s.e) * rate;
    const float move = e2 * em1;                          // e' * (P[b+1]/P[b] - 1)
    pnl = (move - cost) - cost * move;                    // (1 - cost)(1 + move) - 1
    const float V2 = s.V + s.V * pnl;
    s.k += 1;
    const float cpl = V2 - 1.0f;
    label = (cpl >= c.barrier) ? 1 : ((cpl <= -c.barrier) ? -1 : 0);
    done = (label != 0) || (s.k >= c.max_hold);
    v_post = V2;
    if (done) {
        s.V = 1.0f;
        s.e = 0.0f;
        s.k = 0;
    } else {
        s.V = V2;
        s.e = e2;
    }
}

// The rest of the step: the diversity window of categories takes action a's
// category, and the reward combines the trade's pnl and label with the window's
// penalty and the risk term.  Resets the window on done.
__device__ __forceinline__ float env_window_reward(EpState &s, int a, float pnl, int label, int done,
                                                   const EnvConst &c)
{
    const int xi = a / 9;
    const float e2 = 0.5f * (float)(xi - 2);
    // diversity window of categories (Short 0 / Flat 1 / Long 2)
    const int cat = (xi <= 1) ? 0 : ((xi == 2) ? 1 : 2);
    const int W = c.div_window;
    if (s.nwin == W) {
        const int old = (int)((s.win >> (2 * (W - 1))) & 3u);
        s.hist -= hist_unit(old);
        s.nwin -= 1;
    }
    s.win = ((s.win << 2) | (uint64_t)cat) & ((W >= 32) ? ~0ull : ((1ull << (2 * W)) - 1ull));
    s.hist += hist_unit(cat);
    s.nwin += 1;
    // H < threshold, decided exactly (in double, on the host, per histogram)
    const uint32_t bit = s.hist;
    const bool low = (c.div_low[bit >> 5] >> (bit & 31u)) & 1u;   // global or a shared-memory copy
    const float div = low ? c.div_penalty : 0.0f;
    const float beta = (label > 0) ? c.pt_scale : ((label < 0) ? c.sl_scale : 0.0f);
    const float reward = pnl * (1.0f + beta) + div - c.risk_coef * fabsf(e2);
    if (done) {
        s.nwin = 0;
        s.win = 0;
        s.hist = 0;
    }
    return reward;
}

// One environment step for action a; f0_next = F[b+1, 0].  Returns the reward
// without the curiosity bonus; sets v_post = V' and done.  Updates s (including
// the reset on done).
__device__ __forceinline__ float env_step(EpState &s, int a, float f0_next, const EnvConst &c,
                                          float &v_post, int &done)
{
    float pnl;
    int label;
    env_trade(s, a, expm1f(f0_next), c, pnl, v_post, label, done);
    return env_window_reward(s, a, pnl, label, done, c);
}

// exposure held entering step t, recovered from the previous step's action/done
__device__ __forceinline__ float exposure_of(int a) { return 0.5f * (float)(a / 9 - 2); }

__device__ __forceinline__ void set_status(int *status, int code)
{
    atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool start_ok(int start, int L, int n_bars)
{
    return start >= 0 && (long long)start + L <= (long long)n_bars - 1;
}

}  // namespace rl
