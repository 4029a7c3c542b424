// phase1_umma.cu -- tensor-core rollout (phase 1) for ROLLOUT_BF16 / _TF32.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A steps 1-4 and 6-12.  The pages map one
// thread to one episode and run the actor as scalar mat-vecs.  Here a CTA owns
// 128 episodes and runs every actor layer of a step as one M=128 tcgen05 MMA
// (54->128, 128->64, 64->45 padded to 48) with the f32 accumulators in tensor
// memory: thread i of the CTA is episode i, TMEM lane i and A-operand row i.
// The actor weights stay resident in shared memory for the whole rollout.
// Each layer's epilogue (bias, ReLU, rounding to the operand format) is done
// by the owning thread straight from TMEM into the next layer's swizzled
// operand tile; the logits never leave registers: softmax, CDF, LCG draw and
// the environment step follow in the same thread.
#include "env.cuh"
#include "umma.cuh"
#include "umma_path.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kP1Threads = 128;

template <bool BF16>
struct P1Geo {
    static constexpr int EB = BF16 ? 2 : 4;          // bytes per operand element
    static constexpr int KC = 128 / EB;              // elements per K-chunk
    static constexpr int XC = (kState + KC - 1) / KC;    // K-chunks of the state (54 padded)
    static constexpr int H1C = kActorH1 / KC;
    static constexpr int H2C = kActorH2 / KC;
    static constexpr int SLOT = 128 * 128;           // one 128-row K-chunk tile
    static constexpr int IMG = (kActorH1 * XC + kActorH2 * H1C + 48 * H2C) * 128;
    static constexpr int X_OFF = IMG;                // image size is a multiple of 1024
    static constexpr int H1_OFF = X_OFF + XC * SLOT;
    static constexpr int H2_OFF = H1_OFF + H1C * SLOT;
    static constexpr int BIAS_OFF = H2_OFF + H2C * SLOT;
    static constexpr int DIV_OFF = BIAS_OFF + 1024;          // diversity table (kDivWords words)
    // bf16: ring of the market-feature rows of three consecutive steps, one
    // padded row (kFPad floats) per episode, filled by tensor gathers; tf32
    // has no room for it and loads each row thread by thread
    // Layout of a slot: per warp 8 groups of 4 rows, a group (one gather of
    // 4 x 208 B) starting every 896 bytes -- a tensor copy's shared-memory
    // destination must be 128-byte aligned
    static constexpr bool STAGE_F = BF16;
    static constexpr int FR_OFF = DIV_OFF + kDivWords * 4;   // 1024-aligned
    static constexpr int FR_GROUP = 896;
    static constexpr int FR_WARP = 8 * FR_GROUP;
    static constexpr int FR_SLOT = 4 * FR_WARP;
    static constexpr int FR_BYTES = STAGE_F ? 3 * FR_SLOT : 0;
    static constexpr int SMEM = FR_OFF + FR_BYTES + 1024;   // + alignment slack
};

static_assert(P1Geo<true>::FR_OFF % 1024 == 0 && P1Geo<true>::FR_GROUP % 128 == 0 &&
                  P1Geo<true>::FR_GROUP >= 4 * kFPad * 4 && P1Geo<true>::SMEM <= 232448,
              "row ring: 128-byte aligned gather destinations, fits in shared memory");

// write values v[0..n) (n multiple of 8 for bf16, 4 for tf32) as row `r` of a
// K-major swizzled operand starting at column c0 (c0 a multiple of 8 / 4)
template <bool BF16, int N>
__device__ __forceinline__ void put_row(uint8_t *op, int r, int c0, const float (&v)[N])
{
    constexpr int KC = P1Geo<BF16>::KC;
    if constexpr (BF16) {
#pragma unroll
        for (int q = 0; q < N / 8; ++q) {
            const int c = c0 + 8 * q;
            uint4 p;
            p.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
            p.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
            p.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
            p.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
            uint8_t *tile = op + (c / KC) * (128 * 128);
            *reinterpret_cast<uint4 *>(tile + sw128_offset(r, (c % KC) / 8)) = p;
        }
    } else {
#pragma unroll
        for (int q = 0; q < N / 4; ++q) {
            const int c = c0 + 4 * q;
            uint4 p;
            p.x = to_tf32(v[4 * q + 0]);
            p.y = to_tf32(v[4 * q + 1]);
            p.z = to_tf32(v[4 * q + 2]);
            p.w = to_tf32(v[4 * q + 3]);
            uint8_t *tile = op + (c / KC) * (128 * 128);
            *reinterpret_cast<uint4 *>(tile + sw128_offset(r, (c % KC) / 4)) = p;
        }
    }
}

// issue D = A * B^T over `chunks` K-chunks; A tiles are 128 rows, B tiles `nrows` rows
template <bool BF16>
__device__ __forceinline__ void issue_layer(uint32_t d, uint32_t a_base, uint32_t b_base, int chunks, int nrows)
{
    const uint32_t id = idesc(BF16, 128, nrows);
    for (int c = 0; c < chunks; ++c) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint64_t ad = desc_sw128(a_base + c * (128 * 128) + 32 * k);
            const uint64_t bd = desc_sw128(b_base + c * (nrows * 128) + 32 * k);
            mma<BF16>(d, ad, bd, id, (c | k) != 0);
        }
    }
}

// relu(D[col0 .. col0+32*G) + bias) of this thread's lane, into operand `op`
template <bool BF16, int G>
__device__ __forceinline__ void epi_hidden(uint32_t taddr, const float *bias, uint8_t *op, int r)
{
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float v[32];
        tmem_ld32(taddr + 32 * g, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = fmaxf(v[i] + bias[32 * g + i], 0.f);
        put_row<BF16, 32>(op, r, 32 * g, v);
    }
}

template <bool BF16>
__global__ void __launch_bounds__(kP1Threads, 1) phase1_umma_kernel(Phase1Args a, UmmaWeights w,
                                                                    const __grid_constant__ CUtensorMap fmap)
{
    using G = P1Geo<BF16>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *img = sm;
    uint8_t *X = sm + G::X_OFF;
    uint8_t *H1 = sm + G::H1_OFF;
    uint8_t *H2 = sm + G::H2_OFF;
    float *bias = reinterpret_cast<float *>(sm + G::BIAS_OFF);
    uint32_t *sdiv = reinterpret_cast<uint32_t *>(sm + G::DIV_OFF);
    uint8_t *fring = sm + G::FR_OFF;                             // [3][128][kFPad] f32
    __shared__ __align__(8) uint64_t bar_img, bar_mma, bar_final, bar_rows[3];
    __shared__ int s_row0[kP1Threads];                           // bar of step 0 (0 for an episode without rows)
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5;
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_img, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_final, 1);
        for (int k = 0; k < 3; ++k) mbar_init(&bar_rows[k], kP1Threads / 32);   // one arrival per warp
        fence_mbar_init();
    }
    for (int i = tid; i < kActorH1 + kActorH2 + 48; i += kP1Threads) bias[i] = w.actor_bias[i];
    for (int i = tid; i < kDivWords; i += kP1Threads) sdiv[i] = a.env.div_low[i];
    EnvConst env = a.env;
    env.div_low = sdiv;                        // the environment step reads its table from shared memory
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, 256);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int *abort = &abort_sh;

    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_img, w.actor_img_bytes);
        for (uint32_t off = 0; off < w.actor_img_bytes; off += 16384) {
            const uint32_t n = min(16384u, w.actor_img_bytes - off);
            bulk_g2s(img + off, w.actor_img + off, n, &bar_img);
        }
    }
    bool ok = mbar_wait(&bar_img, 0, abort);

    const int n = blockIdx.x * kP1Threads + tid;
    const bool live = n < a.N;
    const int L = a.L;
    const long long row0 = (long long)n * L;
    const int start = live ? a.starts[n] : 0;
    const bool valid = live && start_ok(start, L, a.n_bars);
    if (live && !valid) set_status(a.status, ROLLOUT_ERR_RANGE);
    EpState st;
    ep_reset(st);
    st.rng = live ? a.seeds[n] : 0u;
    const float *F = a.F;
    const int lane = tid & 31;
    s_row0[tid] = valid ? start : 0;
    __syncwarp();
    // bf16: lane 0 of each warp gathers the feature rows of step s (bar
    // start + s; row 0 for an episode without rows) of the warp's 32 episodes
    // into ring slot s % 3 -- eight tensor gathers of four padded rows --
    // two steps ahead of their use; the slot's barrier counts one arrival per warp
    int issued = -1;                                             // last step whose rows were issued
    auto issue_rows = [&](int s) {
        if constexpr (G::STAGE_F) {
            if (s > L) return;
            if (lane == 0) {
                uint64_t *bar = &bar_rows[s % 3];
                uint8_t *dst = fring + (s % 3) * G::FR_SLOT + warp * G::FR_WARP;
                fence_async_smem();                              // the slot's previous rows were read before
                mbar_arrive_expect_tx(bar, 32 * kFPad * 4);
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const int *r0 = s_row0 + warp * 32 + 4 * g;
                    tma_gather4(dst + g * G::FR_GROUP, &fmap, 0, r0[0] + s, r0[1] + s, r0[2] + s, r0[3] + s, bar);
                }
            }
            issued = s;
        }
    };
    // all threads: the rows of step s have landed
    auto wait_rows = [&](int s, volatile int *ab, uint64_t limit) -> bool {
        return mbar_wait(&bar_rows[s % 3], (uint32_t)((s / 3) & 1), ab, limit);
    };

    const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
    const uint32_t sX = smem_u32(X), sH1 = smem_u32(H1), sH2 = smem_u32(H2), sImg = smem_u32(img);
    uint32_t ph = 0;
    float cur[G::STAGE_F ? 1 : kMarket];
    if constexpr (G::STAGE_F) {
        issue_rows(0);
        issue_rows(1);
    } else {
#pragma unroll
        for (int j = 0; j < kMarket; ++j) cur[j] = valid ? __ldg(F + (long long)start * kMarket + j) : 0.f;
    }
    int waited = -1;                                             // last step whose rows were waited for

    ok = __syncthreads_and(ok);
    for (int t = 0; t < L; ++t) {
        // this thread's row in a slot: group lane/4 of its warp, row lane%4 (16-byte aligned)
        const int row_off = warp * G::FR_WARP + (lane >> 2) * G::FR_GROUP + (lane & 3) * kFPad * 4;
        const float4 *row_t = reinterpret_cast<const float4 *>(fring + (t % 3) * G::FR_SLOT + row_off);
        const float *row_n = reinterpret_cast<const float *>(fring + ((t + 1) % 3) * G::FR_SLOT + row_off);
        if constexpr (G::STAGE_F) {
            ok = ok && wait_rows(t, abort, 2000000000ull) && wait_rows(t + 1, abort, 2000000000ull);
            waited = t + 1;
        }
        // state row -> operand X
        {
            float x[G::XC * G::KC];
            if constexpr (G::STAGE_F) {
#pragma unroll
                for (int k = 0; k < kFPad / 4; ++k) {
                    const float4 v = row_t[k];
                    x[4 * k + 0] = valid ? v.x : 0.f;
                    x[4 * k + 1] = valid ? v.y : 0.f;
                    x[4 * k + 2] = valid ? v.z : 0.f;
                    if (4 * k + 3 < kMarket) x[4 * k + 3] = valid ? v.w : 0.f;
                }
            } else {
#pragma unroll
                for (int j = 0; j < kMarket; ++j) x[j] = cur[j];
            }
            x[kMarket] = st.V;
            x[kMarket + 1] = st.e;
            x[kMarket + 2] = a.env.spread;
#pragma unroll
            for (int j = kState; j < G::XC * G::KC; ++j) x[j] = 0.f;
            put_row<BF16, G::XC * G::KC>(X, tid, 0, x);
        }
        // next bar's features: its log-return drives this step, its row is the next state
        float nxt[G::STAGE_F ? 1 : kMarket];
        if constexpr (G::STAGE_F) {
            nxt[0] = valid ? row_n[0] : 0.f;
        } else {
            const long long b = (long long)start + t;
#pragma unroll
            for (int j = 0; j < kMarket; ++j) nxt[j] = valid ? __ldg(F + (b + 1) * kMarket + j) : 0.f;
        }

        fence_async_smem();
        tc_fence_before();
        if (!__syncthreads_and(ok)) break;      // CTA-uniform exit after a failed wait
        tc_fence_after();
        if (tid == 0) {
            issue_layer<BF16>(tmem + 0, sX, sImg + w.actor_off[0], G::XC, kActorH1);
            mma_commit(&bar_mma);
        }
        issue_rows(t + 2);          // slot (t+2)%3 held step t-1's rows, all read before the barrier above
        ok = ok && mbar_wait(&bar_mma, ph, abort);
        ph ^= 1;
        tc_fence_after();
        epi_hidden<BF16, kActorH1 / 32>(lane_addr + 0, bias, H1, tid);

        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            issue_layer<BF16>(tmem + 128, sH1, sImg + w.actor_off[1], G::H1C, kActorH2);
            mma_commit(&bar_mma);
        }
        ok = ok && mbar_wait(&bar_mma, ph, abort);
        ph ^= 1;
        tc_fence_after();
        epi_hidden<BF16, kActorH2 / 32>(lane_addr + 128, bias + kActorH1, H2, tid);

        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            issue_layer<BF16>(tmem + 192, sH2, sImg + w.actor_off[2], G::H2C, 48);
            mma_commit(&bar_mma);
        }
        ok = ok && mbar_wait(&bar_mma, ph, abort);
        ph ^= 1;
        tc_fence_after();
        float logits[kActions];
        {
            float v0[32], v1[32];
            tmem_ld32(lane_addr + 192, v0);
            tmem_ld32(lane_addr + 224, v1);
            tmem_ld_wait();
            const float *b3 = bias + kActorH1 + kActorH2;
#pragma unroll
            for (int j = 0; j < 32; ++j) logits[j] = v0[j] + b3[j];
#pragma unroll
            for (int j = 32; j < kActions; ++j) logits[j] = v1[j - 32] + b3[j];
        }
        const float u = lcg_uniform(st.rng);
        float logp;
        const int act = sample_action<kActions>(logits, u, logp);
        const float v_in = st.V;
        float v_post;
        int done;
        const float rew = env_step(st, act, nxt[0], env, v_post, done);
        if (valid && ok) {
            a.actions[row0 + t] = act;
            a.logp[row0 + t] = logp;
            a.dones[row0 + t] = done;
            a.rewards[row0 + t] = rew;
            a.v_in[row0 + t] = v_in;
            a.v_post[row0 + t] = v_post;
        } else if (live) {
            a.actions[row0 + t] = 0;
            a.logp[row0 + t] = 0.f;
            a.dones[row0 + t] = 0;
            a.rewards[row0 + t] = 0.f;
            a.v_in[row0 + t] = 0.f;
            a.v_post[row0 + t] = 0.f;
        }
        if constexpr (!G::STAGE_F) {
#pragma unroll
            for (int j = 0; j < kMarket; ++j) cur[j] = nxt[j];
        }
    }
    if constexpr (G::STAGE_F) {
        // rows still in flight after an early exit land before the CTA ends
        // (bounded waits that do not give up on the abort flag)
        int never = 0;
        for (int s = waited + 1; s <= issued; ++s) wait_rows(s, &never, 100000000ull);
    }
    if (tid == 0) {
        if (!ok) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
        // every MMA issued must complete before TMEM is released (bounded wait)
        mma_commit(&bar_final);
        int never = 0;
        mbar_wait(&bar_final, 0, &never, 100000000ull);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, 256);
}

template <bool BF16>
cudaError_t launch_p1(const Phase1Args &a, const UmmaWeights &w, const CUtensorMap &fmap, cudaStream_t s)
{
    using G = P1Geo<BF16>;
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(phase1_umma_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             G::SMEM);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    const int blocks = (a.N + kP1Threads - 1) / kP1Threads;
    phase1_umma_kernel<BF16><<<blocks, kP1Threads, G::SMEM, s>>>(a, w, fmap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_phase1_umma(const Phase1Args &a, const UmmaWeights &w, const CUtensorMap &fmap, cudaStream_t s)
{
    return w.bf16 ? launch_p1<true>(a, w, fmap, s) : launch_p1<false>(a, w, fmap, s);
}

namespace {

// the feature matrix with rows padded to kFPad floats (the extra column is
// zero): a tensor map's row pitch must be a multiple of 16 bytes, 51 floats
// (204 bytes) is not
__global__ void pad_features_kernel(const float *F, float4 *P, long long n_bars)
{
    constexpr int W = kFPad / 4;                 // 16-byte words per padded row
    const long long total = n_bars * W;
    for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < total;
         i += (long long)gridDim.x * blockDim.x) {
        const long long b = i / W;
        const int c0 = 4 * (int)(i - b * W);
        float v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) v[j] = c0 + j < kMarket ? __ldg(F + b * kMarket + c0 + j) : 0.f;
        P[i] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

}  // namespace

cudaError_t launch_pad_features(const float *F, float *fpad, int n_bars, cudaStream_t s)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long words = (long long)n_bars * (kFPad / 4);
    const long long blocks = (words + 255) / 256;
    const int grid = (int)(blocks < (long long)sms * 8 ? blocks : (long long)sms * 8);
    pad_features_kernel<<<grid, 256, 0, s>>>(F, reinterpret_cast<float4 *>(fpad), n_bars);
    return cudaGetLastError();
}

}  // namespace rl
