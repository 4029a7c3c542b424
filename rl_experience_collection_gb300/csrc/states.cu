// states.cu -- the stored state rows s_t = [F[bar_t, 0:51], V_t, e_t, spread]
// of every tuple, written to out_states [N, L, 54] (f32, row-major).
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A step 3 (the 54-wide state: 51 market
// features + 3 portfolio features) and step 11 (the tuple is stored); page
// "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA Experience Collection", section
// "Kernel Components" 3 (portfolio features).
//
// Runs after the rollout kernel and before the value phase, while out_values
// still holds V_t, the portfolio value entering each step.  e_t is 0 at t = 0
// and after a reset, else the exposure of a_{t-1}.  Every row of an episode
// whose start bar is out of range is zero.
//
// Each warp owns chunks of 32 consecutive rows: its lanes resolve one row's
// metadata each, then the warp writes the chunk row by row, lane l storing
// columns l and 32 + l (l < 22), so that every store instruction covers a
// contiguous run of the row.  Warps synchronise only with themselves, so
// many chunks are in flight per SM, and the feature loads of 8 rows are
// issued before their stores.  The market columns come from the feature
// matrix, which is small enough to stay in L2.
#include "env.cuh"

namespace rl {

namespace {

constexpr int kWarps = 8;
constexpr int kBatchRows = 16;

__global__ void __launch_bounds__(kWarps * 32) states_kernel(StatesArgs a)
{
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const long long NL = (long long)a.N * a.L;
    const long long n_chunks = (NL + 31) / 32;
    const bool narrow = NL <= 0x7fffffffLL;
    const int c1 = 32 + lane;                     // the lane's column in the row's second part
    for (long long ch = (long long)blockIdx.x * kWarps + wi; ch < n_chunks; ch += (long long)gridDim.x * kWarps) {
        const long long row0 = ch * 32, row = row0 + lane;
        long long fb = -1;                        // float offset of the row's bar in F, or -1: zero row
        float v = 0.f, e = 0.f;
        if (row < NL) {
            long long n;
            if (narrow) n = (long long)((uint32_t)row / (uint32_t)a.L);
            else n = row / a.L;
            const int t = (int)(row - n * a.L);
            const int start = __ldg(a.starts + n);
            const float vin = a.v_in[row];
            const int dprev = t > 0 ? a.dones[row - 1] : 1;
            const int aprev = t > 0 ? a.actions[row - 1] : 0;
            if (start_ok(start, a.L, a.n_bars)) {
                fb = ((long long)start + t) * kMarket;
                v = vin;
                e = dprev ? 0.f : exposure_of(aprev);
            }
        }
        const int n_rows = NL - row0 < 32 ? (int)(NL - row0) : 32;
        float *dst = a.states + row0 * kState;
#pragma unroll 1
        for (int r0 = 0; r0 < 32; r0 += kBatchRows) {
            float x0[kBatchRows], x1[kBatchRows];
#pragma unroll
            for (int k = 0; k < kBatchRows; ++k) {
                const long long f = __shfl_sync(0xffffffffu, fb, r0 + k);
                const float vv = __shfl_sync(0xffffffffu, v, r0 + k);
                const float ee = __shfl_sync(0xffffffffu, e, r0 + k);
                float y0 = 0.f, y1 = 0.f;
                if (f >= 0) {
                    y0 = __ldg(a.F + f + lane);
                    if (c1 < kMarket) y1 = __ldg(a.F + f + c1);
                    else if (c1 == kMarket) y1 = vv;
                    else if (c1 == kMarket + 1) y1 = ee;
                    else if (c1 == kMarket + 2) y1 = a.spread;
                }
                x0[k] = y0;
                x1[k] = y1;
            }
#pragma unroll
            for (int k = 0; k < kBatchRows; ++k) {
                const int rr = r0 + k;
                if (rr < n_rows) {
                    __stcs(dst + rr * kState + lane, x0[k]);
                    if (c1 < kState) __stcs(dst + rr * kState + c1, x1[k]);
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_states(const StatesArgs &a, cudaStream_t s)
{
    const long long NL = (long long)a.N * a.L;
    const long long blocks = ((NL + 31) / 32 + kWarps - 1) / kWarps;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long cap = (long long)sms * 16;
    const int grid = (int)(blocks < cap ? blocks : cap);
    states_kernel<<<grid, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace rl
