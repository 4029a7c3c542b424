// gae.cu -- backward GAE as a warp-parallel segmented linear recurrence.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase B:
//   delta_t = r_t + gamma * V_{t+1} * (1 - d_t) - V_t      (V_L = bootstrap)
//   A_t     = delta_t + gamma * lambda * (1 - d_t) * A_{t+1} (A_L = 0)
//   R_t     = A_t + V_t
// The pages scan each episode sequentially in one thread.  Here one warp owns
// an episode and walks it backwards in chunks of 32 steps: each lane holds the
// affine map A -> delta_t + c_t * A (c_t = gamma*lambda*(1-d_t)); a Kogge-Stone
// suffix scan composes the maps inside the chunk ((c1,d1) o (c2,d2) =
// (c1*c2, d1 + c1*d2)) and the chunk's A_{t0} is carried to the next chunk.
// Reads r, V, d and writes A, R with coalesced 128-byte warp accesses.
#include "internal.cuh"

namespace rl {

namespace {

constexpr int kGaeWarps = 8;

__global__ void __launch_bounds__(kGaeWarps * 32) gae_kernel(GaeArgs a)
{
    const int lane = threadIdx.x & 31;
    const int n = blockIdx.x * kGaeWarps + (threadIdx.x >> 5);
    if (n >= a.N) return;
    const int L = a.L;
    const long long base = (long long)n * L;
    const float gl = a.gamma * a.lambda;
    float carry_adv = 0.0f;                              // A_{t0+32}
    float carry_v = a.ret[base + L - 1];                 // V_{t0+32}: bootstrap first
    const int n_chunks = (L + 31) / 32;
    for (int c = n_chunks - 1; c >= 0; --c) {
        const int t = c * 32 + lane;
        const bool live = t < L;
        const float r = live ? a.rewards[base + t] : 0.f;
        const float v = live ? a.values[base + t] : 0.f;
        const int d = live ? a.dones[base + t] : 0;
        // V_{t+1}: next lane, or the carried value for the chunk's last live step
        float v_next = __shfl_down_sync(0xffffffffu, v, 1);
        const int last_live = min(31, L - 1 - c * 32);
        if (lane == last_live) v_next = carry_v;
        const float nd = d ? 0.f : 1.f;
        float dl = live ? (r + a.gamma * v_next * nd - v) : 0.f;
        float cc = live ? gl * nd : 1.f;
        // inclusive suffix scan of affine maps over lanes lane..31
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float dl_o = __shfl_down_sync(0xffffffffu, dl, off);
            const float cc_o = __shfl_down_sync(0xffffffffu, cc, off);
            if (lane + off < 32) {
                dl = fmaf(cc, dl_o, dl);
                cc = cc * cc_o;
            }
        }
        const float A = fmaf(cc, carry_adv, dl);
        if (live) {
            a.adv[base + t] = A;
            a.ret[base + t] = A + v;
        }
        carry_adv = __shfl_sync(0xffffffffu, A, 0);
        carry_v = __shfl_sync(0xffffffffu, v, 0);
    }
}

}  // namespace

cudaError_t launch_gae(const GaeArgs &a, cudaStream_t s)
{
    const int blocks = (a.N + kGaeWarps - 1) / kGaeWarps;
    gae_kernel<<<blocks, kGaeWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace rl
