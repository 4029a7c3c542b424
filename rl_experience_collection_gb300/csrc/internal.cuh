// internal.cuh -- declarations shared by the translation units of librollout.
//
// The collector runs as stream-ordered phases, with no host round trip:
//   phase 1 (rollout): per episode, per step: actor MLP, softmax/CDF/LCG
//     sample, portfolio, triple-barrier and diversity step, reset on done.
//     The critic and the curiosity model do not feed the state trajectory,
//     so they are not on this serial chain.
//   state rows: every tuple's stored state row (states.cu).
//   phase 2 (value): every tuple independently (plus one bootstrap row per
//     episode): rebuilds the state row, runs the critic MLP and the curiosity
//     model, adds the curiosity bonus to the reward.
//   phase 3 (gae): per episode, a warp-parallel segmented backward scan.
// Between the phases the outputs double as intermediate storage:
//   out_values[n,t] holds the portfolio value V entering step t (phase 1 ->
//   phase 2, which overwrites it with the critic value), out_adv[n,t] holds
//   the post-trade value V' (phase 1 -> phase 2, overwritten by phase 3),
//   out_ret[n,L-1] holds the bootstrap value (phase 2 -> phase 3).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/rollout.h"

namespace rl {

// environment constants, passed by value to the kernels
struct EnvConst {
    float barrier;
    int max_hold;
    float pt_scale, sl_scale;
    int div_window;
    float div_thresh, div_penalty;
    float cur_coef, risk_coef, tx_base, spread;
    // bit (c0*1024 + c1*32 + c2): 1 when the Shannon entropy (bits) of the
    // category histogram (c0, c1, c2) is below div_thresh; 32768 bits
    // (kDivWords words); kernels may point this at a shared-memory copy
    const uint32_t *div_low;
};

constexpr int kDivWords = 1024;
constexpr int kMarket = 51;
constexpr int kFPad = 52;          // padded feature row (208 bytes, a multiple of 16) for tensor maps
constexpr int kState = 54;
constexpr int kActions = 45;
constexpr int kActorH1 = 128;
constexpr int kActorH2 = 64;
constexpr int kCurH = 64;
constexpr int kCriticLayers = 6;   // 5 hidden + scalar head

// Test hook (rollout_test_activations): the rounded operands that the
// tensor-core kernels feed to their layers, for the first n_ep episodes.
// Row n*(L+1)+t holds step t of episode n, row n*(L+1)+L the bootstrap critic
// of episode n; a row is `width` floats: state input (kDumpIn columns, the
// first kState used) | actor h1 (from act_off) | actor h2 | critic hidden
// layers (crit_off[l] is layer l's first column) | curiosity hidden (from
// cur_off).  p == nullptr: nothing is written (the normal builds of the
// kernels never write it).
constexpr int kDumpIn = 64;
struct ActDump {
    float *p = nullptr;
    int n_ep = 0;
    int width = 0;
    int act_off = kDumpIn;
    int crit_off[5] = {};
    int cur_off = 0;
    // row of step t of episode n (t == L: its bootstrap row), or nullptr
    __device__ __forceinline__ float *row(long long n, int t, int L) const
    {
        return (p && n >= 0 && n < n_ep) ? p + ((long long)n * (L + 1) + t) * width : nullptr;
    }
};

// ReLU as max(x, 0) through the comparison x < 0: a NaN input stays NaN (as
// with cvt.rn.relu), where fmaxf(x, 0) would turn it into 0
__device__ __forceinline__ float relu(float x) { return x < 0.f ? 0.f : x; }

// device status word values (first error wins)
constexpr int kStatusOk = 0;

struct Phase1Args {
    const float *F;            // [n_bars, 51]
    const int32_t *starts;     // [N]
    const uint32_t *seeds;     // [N]
    int N, L, n_bars;
    int32_t *actions;          // [N, L]
    float *logp;               // [N, L]
    int32_t *dones;            // [N, L]
    float *rewards;            // [N, L]: reward without the curiosity bonus
    float *v_in;               // [N, L]: V entering the step (out_values)
    float *v_post;             // [N, L]: V' after the trade (out_adv)
    int *status;
    EnvConst env;
    ActDump dump;              // test hook, see ActDump
};

struct ValueArgs {
    const float *F;
    const int32_t *starts;
    int N, L, n_bars;
    const int32_t *actions;
    const int32_t *dones;
    float *values;             // in: V entering the step; out: critic value
    const float *v_post;       // V' after the trade
    float *rewards;            // in: base reward; out: + curiosity bonus
    float *boot;               // out_ret: [n*L + L-1] receives the bootstrap value
    int *status;
    EnvConst env;
    ActDump dump;              // test hook, see ActDump
};

// the stored state rows (states.cu), written between the rollout and the value phase
struct StatesArgs {
    const float *F;
    const int32_t *starts;
    int N, L, n_bars;
    const int32_t *actions;
    const int32_t *dones;
    const float *v_in;         // V entering each step (out_values before the value phase)
    float spread;
    float *states;             // [N, L, 54] written
    const float *Fpad = nullptr;   // optional copy of F with rows padded to kFPad floats (16-byte aligned rows)
    const int32_t *bars = nullptr; // optional bar of every step (episode recycling); else start + t
};

// the feature matrix with rows padded to kFPad floats (16-byte aligned rows;
// column 51 holds the bar's simple return expm1(F[b, 0])), for 16-byte loads
// and tensor maps (phase1_umma.cu)
cudaError_t launch_pad_features(const float *F, float *fpad, int n_bars, cudaStream_t s);

struct GaeArgs {
    const float *rewards, *values;
    const int32_t *dones;
    float *adv, *ret;          // ret[n*L + L-1] holds the bootstrap value on entry
    int N, L;
    float gamma, lambda;
};

// --- float32 CUDA-core path (simt.cu) ---
struct SimtWeights {
    const float *actor;        // per layer: W^T [in][out_pad4] then b[out]; see api.cu
    const float *critic_T[kCriticLayers];   // W^T [in][out]
    const float *critic_b[kCriticLayers];
    int critic_w[kCriticLayers + 1];         // widths: in, h1..h5, 1
    const float *cur0_T, *cur0_b;           // [99][64], [64]
    const float *cur1_T, *cur1_b;           // [64][54], [54]
};
cudaError_t launch_phase1_simt(const Phase1Args &a, const float *actor_packed, cudaStream_t s);
cudaError_t launch_value_simt(const ValueArgs &a, const SimtWeights &w, cudaStream_t s);

// --- state rows (states.cu) ---
cudaError_t launch_states(const StatesArgs &a, cudaStream_t s);

// --- GAE (gae.cu) ---
cudaError_t launch_gae(const GaeArgs &a, cudaStream_t s);

// Runs set_up() (a kernel's attribute calls) once per device, on the current
// device, and remembers which devices are done; devices past 63 run it on
// every call.  Returns its status.
template <class F>
inline cudaError_t once_per_device(std::atomic<unsigned long long> &done, F &&set_up)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 64) return set_up();
    const unsigned long long bit = 1ull << dev;
    if (done.load() & bit) return cudaSuccess;
    e = set_up();
    if (e == cudaSuccess) done.fetch_or(bit);
    return e;
}

// --- device allocations of rollout handles (api.cu) ---
// Every device allocation a rollout handle makes goes through dev_alloc /
// dev_free, which count the live ones and let a test make the k-th
// allocation fail as if the device were out of memory (rollout_test_alloc).
cudaError_t dev_alloc(void **p, size_t bytes);
void dev_free(void *p);

// --- shared host helpers (api.cu) ---
int set_error(int code, const char *fmt, ...);   // records the message rollout_last_error returns; returns code
void clear_error();
int validate_dims(const rollout_dims *d);         // the shapes rollout_create accepts

}  // namespace rl
