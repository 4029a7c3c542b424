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
// and after a reset, else the exposure of a_{t-1}.  bar_t is start + t, or the
// bar the rollout stored for the step (the DQN collector's episode recycling).
// Every row of an episode whose start bar is out of range is zero.
//
// Each warp owns chunks of 32 consecutive rows (6912 bytes, 54 whole 128-byte
// lines of out_states): its lanes resolve one row's metadata each into shared
// memory, then the warp writes the chunk as a flat run of 864 float pairs, lane
// l storing pairs l, l + 32, ... -- a pair never straddles two rows (54 is
// even), and every store instruction covers two whole lines.  Pairs 0..24 of a
// row are market features, pair 25 is (F[.., 50], V), pair 26 is (e, spread).
// The feature loads of three pairs are issued before their stores.  The market
// columns come from the feature matrix, which is small enough to stay in L2;
// where the padded copy (rows of kFPad floats, 16-byte aligned) exists, each
// pair is one 8-byte load, which halves the loads the L1 has in flight.
#include "env.cuh"

namespace rl {

namespace {

constexpr int kWarps = 32;
constexpr int kPairs = kState / 2;            // 27 float pairs per row
constexpr int kBatch = 3;                     // pairs per lane with loads in flight (more warps beat deeper batches)

template <bool PAD>
__global__ void __launch_bounds__(kWarps * 32) states_kernel(StatesArgs a)
{
    constexpr int RS = PAD ? kFPad : kMarket;  // row stride of the feature source
    const float *src = PAD ? a.Fpad : a.F;
    __shared__ long long s_fb[kWarps][32];    // float offset of the row's bar in the source, or -1: zero row
    __shared__ float2 s_ve[kWarps][32];       // V, e of the row
    const int lane = threadIdx.x & 31, wi = threadIdx.x >> 5;
    const long long NL = (long long)a.N * a.L;
    const long long n_chunks = (NL + 31) / 32;
    const bool narrow = NL <= 0x7fffffffLL;
    for (long long ch = (long long)blockIdx.x * kWarps + wi; ch < n_chunks; ch += (long long)gridDim.x * kWarps) {
        const long long row0 = ch * 32, row = row0 + lane;
        long long fb = -1;
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
                long long b = (long long)start + t;
                // a stored bar (episode recycling), read where the rollout wrote it
                if (a.bars) {
                    b = a.bars[row];
                    if (b < 0 || b > a.n_bars - 2) b = 0;
                }
                fb = b * RS;
                v = vin;
                e = dprev ? 0.f : exposure_of(aprev);
            }
        }
        __syncwarp();                         // the previous chunk's reads of the slots are done
        s_fb[wi][lane] = fb;
        s_ve[wi][lane] = make_float2(v, e);
        __syncwarp();
        const int n_rows = NL - row0 < 32 ? (int)(NL - row0) : 32;
        const int n_pairs = n_rows * kPairs;
        float2 *dst = reinterpret_cast<float2 *>(a.states + row0 * kState);
#pragma unroll 1
        for (int j0 = 0; j0 < 32 * kPairs; j0 += 32 * kBatch) {
            float2 x[kBatch];
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int j = j0 + 32 * k + lane;
                const int r = j / kPairs, cp = j - kPairs * r;
                float2 y = make_float2(0.f, 0.f);
                if (j < n_pairs) {
                    const long long f = s_fb[wi][r];
                    if (f >= 0) {
                        if (cp < kPairs - 2) {
                            if constexpr (PAD) {
                                y = __ldg(reinterpret_cast<const float2 *>(src + f) + cp);
                            } else {
                                y.x = __ldg(src + f + 2 * cp);
                                y.y = __ldg(src + f + 2 * cp + 1);
                            }
                        } else if (cp == kPairs - 2) {
                            y.x = __ldg(src + f + kMarket - 1);
                            y.y = s_ve[wi][r].x;
                        } else {
                            y.x = s_ve[wi][r].y;
                            y.y = a.spread;
                        }
                    }
                }
                x[k] = y;
            }
#pragma unroll
            for (int k = 0; k < kBatch; ++k) {
                const int j = j0 + 32 * k + lane;
                if (j < n_pairs) __stcs(dst + j, x[k]);
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
    if (a.Fpad) states_kernel<true><<<grid, kWarps * 32, 0, s>>>(a);
    else states_kernel<false><<<grid, kWarps * 32, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace rl
