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
// the environment step follow in the same thread.  The bf16 kernel gives each
// episode four threads instead and takes layer 1's action-independent inputs
// off the serial chain (see phase1_bf16_kernel).
#include <cuda_bf16.h>

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

// the operand values of a packed bf16 unit (8 values) or tf32 unit (4) at dst
__device__ __forceinline__ void dump_unit_bf16(float *dst, uint4 p)
{
    const float2 a = unpack_bf16x2(p.x), b = unpack_bf16x2(p.y), c = unpack_bf16x2(p.z), d = unpack_bf16x2(p.w);
    reinterpret_cast<float4 *>(dst)[0] = make_float4(a.x, a.y, b.x, b.y);
    reinterpret_cast<float4 *>(dst)[1] = make_float4(c.x, c.y, d.x, d.y);
}
__device__ __forceinline__ void dump_unit_tf32(float *dst, uint4 p)
{
    *reinterpret_cast<float4 *>(dst) =
        make_float4(__uint_as_float(p.x), __uint_as_float(p.y), __uint_as_float(p.z), __uint_as_float(p.w));
}

// write values v[0..n) (n multiple of 8 for bf16, 4 for tf32) as row `r` of a
// K-major swizzled operand starting at column c0 (c0 a multiple of 8 / 4);
// D: also the rounded values to dst[0..n) when dst is not null (test hook)
template <bool BF16, int N, bool D = false>
__device__ __forceinline__ void put_row(uint8_t *op, int r, int c0, const float (&v)[N], float *dst = nullptr)
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
            if constexpr (D) {
                if (dst) dump_unit_bf16(dst + 8 * q, p);
            }
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
            if constexpr (D) {
                if (dst) dump_unit_tf32(dst + 4 * q, p);
            }
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
// (D: and to dst[0 .. 32*G) when dst is not null)
template <bool BF16, int G, bool D = false>
__device__ __forceinline__ void epi_hidden(uint32_t taddr, const float *bias, uint8_t *op, int r,
                                           float *dst = nullptr)
{
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float v[32];
        tmem_ld32(taddr + 32 * g, v);
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = relu(v[i] + bias[32 * g + i]);
        put_row<BF16, 32, D>(op, r, 32 * g, v, dst ? dst + 32 * g : nullptr);
    }
}

// kDump: the test build that also writes the rounded hidden activations (ActDump)
template <bool BF16, bool kDump>
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
        float *drow = nullptr;
        if constexpr (kDump) drow = live ? a.dump.row(n, t, L) : nullptr;
        epi_hidden<BF16, kActorH1 / 32, kDump>(lane_addr + 0, bias, H1, tid, drow ? drow + a.dump.act_off : nullptr);

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
        epi_hidden<BF16, kActorH2 / 32, kDump>(lane_addr + 128, bias + kActorH1, H2, tid,
                                                drow ? drow + a.dump.act_off + kActorH1 : nullptr);

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

// ---------------------------------------------------------------------------
// bf16 rollout with four threads per episode.  Warp w serves TMEM lanes and
// episodes 32*(w%4)..+31 (its "quarter") and part p = w/4 of each row: the
// state columns [16p, +16), layer 1's [32p, +32), layer 2's [16p, +16) and
// the logits [12p, +12).
//
// Layer 1 is split by what each input depends on.  The 51 market features,
// the spread and the bias (three bf16 pieces b = hi + mid + lo against three
// constant-one columns 54..56 of the state tile) do not depend on the action
// drawn in the step before, so their MMA for step t+1 runs on the tensor pipe
// while step t samples its action.  The two portfolio inputs V and e (columns
// 51, 52, zero in the MMA operand) enter in the epilogue as
// bf16(V)*W1[:,51] + e*W1[:,52], exact products of bf16 values summed in f32.
// Every part runs the short trade step (V', label, done, the V/e/k update)
// itself from the shared draw, so no exchange closes the step; the step's
// outputs, and on part 3 the diversity window and the reward, which nothing
// else in the step needs, are written one step late while the next step's
// layer 3 is on the tensor pipe.
//
// The softmax is split over the four parts: each takes its block's maximum
// and sum, the blocks are merged (sum_p s_p * exp(m_p - m)), and each part
// scans its block of the index-order CDF from the sum of the blocks before
// it; the lowest part with a crossing gives the action, part 3 taking action
// 44 when round-off leaves u*S above every running sum.
// A 17th warp issues every MMA, so that no worker warp stalls behind the
// tensor pipe's instruction queue, and two more issue the row gathers (tensor
// copies issued by one warp run one after another, at over a hundred cycles
// each).  Barrier 0 (the whole CTA) orders H1 before layer 2 and frees the
// ring slot the loaders refill; barrier 5 (workers and MMA warp) orders H2 and
// the next state tile before layer 3 and layer 1; barriers 1-4 order the
// exchanges inside each quarter.
constexpr int kWorkerWarps = 16;
constexpr int kLoaderWarps = 2;
constexpr int kQThreads = 32 * (kWorkerWarps + 1 + kLoaderWarps);
constexpr int kBarB = 5, kBarBThreads = 32 * (kWorkerWarps + 1);
constexpr int kNone = 99;                      // no crossing in a part's block
// tensor memory columns: layer 1 [0, 128), layer 2 [128, 192), layer 3 [192, 240)
constexpr int kP1TmemCols = 256;
constexpr int kD1 = 0, kD2 = 128, kD3 = 192;
constexpr int kLogitsPerPart = 12;

__device__ __forceinline__ void qsync(int quarter)
{
    asm volatile("bar.sync %0, %1;" ::"r"(1 + quarter), "n"(kP1Threads) : "memory");
}

__device__ __forceinline__ void barrier_b() { asm volatile("bar.sync %0, %1;" ::"n"(kBarB), "n"(kBarBThreads) : "memory"); }

// d = a * b + c on two f32 lanes at once, each rounded as fmaf
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c)
{
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(r)
        : "l"(*reinterpret_cast<uint64_t *>(&a)), "l"(*reinterpret_cast<uint64_t *>(&b)),
          "l"(*reinterpret_cast<uint64_t *>(&c)));
    return *reinterpret_cast<float2 *>(&r);
}

template <int NX>
__device__ __forceinline__ void tmem_ld_x(uint32_t taddr, float *v);

template <>
__device__ __forceinline__ void tmem_ld_x<16>(uint32_t taddr, float *v)
{
    uint32_t x[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
          "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(x[i]);
}

template <>
__device__ __forceinline__ void tmem_ld_x<4>(uint32_t taddr, float *v)
{
    uint32_t x[4];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3])
                 : "r"(taddr)
                 : "memory");
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(x[i]);
}

// relu(v[0..N)) as bf16, row r, columns c0.. of a K-major swizzled operand (c0 % 8 == 0, N % 8 == 0);
// D: also the rounded values to dst[0..N) when dst is not null (test hook)
template <int N, bool D = false>
__device__ __forceinline__ void put_row_relu(uint8_t *op, int r, int c0, const float (&v)[N], float *dst = nullptr)
{
    constexpr int KC = P1Geo<true>::KC;
#pragma unroll
    for (int q = 0; q < N / 8; ++q) {
        const int c = c0 + 8 * q;
        uint4 p;
        p.x = pack_bf16x2_relu(v[8 * q + 0], v[8 * q + 1]);
        p.y = pack_bf16x2_relu(v[8 * q + 2], v[8 * q + 3]);
        p.z = pack_bf16x2_relu(v[8 * q + 4], v[8 * q + 5]);
        p.w = pack_bf16x2_relu(v[8 * q + 6], v[8 * q + 7]);
        uint8_t *tile = op + (c / KC) * (128 * 128);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(r, (c % KC) / 8)) = p;
        if constexpr (D) {
            if (dst) dump_unit_bf16(dst + 8 * q, p);
        }
    }
}

// byte offset of element (row n, column k) in a bf16 K-major swizzled tile
__device__ __forceinline__ uint32_t bf16_elem_offset(int n, int k)
{
    return sw128_offset(n, k >> 3) + 2 * (k & 7);
}

__device__ __forceinline__ float bf16_round(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

// kDump: the test build that also writes the rounded hidden activations (ActDump)
template <bool kDump>
__global__ void __launch_bounds__(kQThreads, 1) phase1_bf16_kernel(Phase1Args a, UmmaWeights w,
                                                                  const __grid_constant__ CUtensorMap fmap)
{
    using G = P1Geo<true>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *img = sm;
    uint8_t *X = sm + G::X_OFF;
    uint8_t *H1 = sm + G::H1_OFF;
    uint8_t *H2 = sm + G::H2_OFF;
    float *bias = reinterpret_cast<float *>(sm + G::BIAS_OFF);   // b2[64] | b3[48]
    uint32_t *sdiv = reinterpret_cast<uint32_t *>(sm + G::DIV_OFF);
    uint8_t *fring = sm + G::FR_OFF;                             // [3] slots, see P1Geo
    __shared__ __align__(8) uint64_t bar_img, bar_l1, bar_mma, bar_final, bar_rows[3];
    __shared__ int s_row0[kP1Threads];                           // start bar (0 for an episode without rows)
    __shared__ __align__(16) float s_wv[kActorH1];               // W1[:, 51] (bf16 values), read as float4
    __shared__ __align__(16) float s_we[kActorH1];               // W1[:, 52]
    __shared__ float2 s_ms[4][kP1Threads];                       // per part: block maximum, block sum
    __shared__ int s_cand[4][kP1Threads];                        // per part: first crossing or kNone
    __shared__ float s_la[4][kP1Threads];                        // its logit
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool issuer = warp == kWorkerWarps;                    // the MMA warp
    const bool leader = issuer && lane == 0;                     // the thread that issues
    const bool loader = warp > kWorkerWarps;                     // the gather warps
    const bool worker = warp < kWorkerWarps;
    const int quarter = warp & 3, part = warp >> 2;
    const int ei = 32 * quarter + lane;                          // episode within the CTA = TMEM lane = MMA row
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_img, 1);
        mbar_init(&bar_l1, 1);
        mbar_init(&bar_mma, 1);
        mbar_init(&bar_final, 1);
        for (int k = 0; k < 3; ++k) mbar_init(&bar_rows[k], kLoaderWarps);   // one arrival per loader warp
        fence_mbar_init();
    }
    for (int i = tid; i < kActorH2 + 48; i += kQThreads) bias[i] = w.actor_bias[kActorH1 + i];
    for (int i = tid; i < kDivWords; i += kQThreads) sdiv[i] = a.env.div_low[i];
    EnvConst env = a.env;
    env.div_low = sdiv;
    if (warp == 0) {
        tmem_alloc(&tmem_base_sh, kP1TmemCols);
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
            const uint32_t nb = min(16384u, w.actor_img_bytes - off);
            bulk_g2s(img + off, w.actor_img + off, nb, &bar_img);
        }
    }
    bool ok = mbar_wait(&bar_img, 0, abort);
    if (tid < kActorH1) {
        // W1 row j: take out the portfolio weights, put the bias pieces at columns 54..56
        uint8_t *w1 = img + w.actor_off[0];
        const int j = tid;
        s_wv[j] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(w1 + bf16_elem_offset(j, kMarket)));
        s_we[j] = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(w1 + bf16_elem_offset(j, kMarket + 1)));
        const float b = w.actor_bias[j];
        const __nv_bfloat16 hi = __float2bfloat16_rn(b);
        const float r1 = b - __bfloat162float(hi);
        const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
        const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
        *reinterpret_cast<__nv_bfloat16 *>(w1 + bf16_elem_offset(j, kState + 0)) = hi;
        *reinterpret_cast<__nv_bfloat16 *>(w1 + bf16_elem_offset(j, kState + 1)) = mid;
        *reinterpret_cast<__nv_bfloat16 *>(w1 + bf16_elem_offset(j, kState + 2)) = lo;
    }

    const int n = blockIdx.x * kP1Threads + ei;
    const bool live = worker && n < a.N;
    const int L = a.L;
    const long long row0 = (long long)n * L;
    const int start = live ? a.starts[n] : 0;
    const bool valid = live && start_ok(start, L, a.n_bars);
    if (part == 0 && live && !valid) set_status(a.status, ROLLOUT_ERR_RANGE);
    EpState st;
    ep_reset(st);
    st.rng = live ? a.seeds[n] : 0u;
    if (part == 0) s_row0[ei] = valid ? start : 0;
    __syncthreads();
    // lane 0 of loader warp k gathers quarters 2k and 2k+1 (16 groups of four
    // rows); every thread tracks `issued`
    int issued = -1;
    auto issue_rows = [&](int s) {
        if (s > L) return;
        if (loader && lane == 0) {
            const int k = warp - kWorkerWarps - 1;
            uint64_t *bar = &bar_rows[s % 3];
            uint8_t *dst = fring + (s % 3) * G::FR_SLOT;
            fence_async_smem();
            mbar_arrive_expect_tx(bar, (kP1Threads / kLoaderWarps) * kFPad * 4);
            for (int g = 16 * k; g < 16 * k + 16; ++g) {
                const int *r0 = s_row0 + 4 * g;
                tma_gather4(dst + (g >> 3) * G::FR_WARP + (g & 7) * G::FR_GROUP, &fmap, 0, r0[0] + s, r0[1] + s,
                            r0[2] + s, r0[3] + s, bar);
            }
        }
        issued = s;
    };
    int waited = -1;
    auto wait_rows = [&](int s) -> bool {
        if (!mbar_wait(&bar_rows[s % 3], (uint32_t)((s / 3) & 1), abort)) return false;
        waited = s;
        return true;
    };
    const int row_off = quarter * G::FR_WARP + (lane >> 2) * G::FR_GROUP + (lane & 3) * kFPad * 4;
    auto ring_row = [&](int s) { return reinterpret_cast<const float4 *>(fring + (s % 3) * G::FR_SLOT + row_off); };
    // state columns [16p, +16) of step s from its feature row; the portfolio
    // columns are zero here, the three bias columns one
    auto build_x = [&](int s) {
        const float4 *row = ring_row(s);
        float x[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 v = row[4 * part + k];
            x[4 * k + 0] = v.x;
            x[4 * k + 1] = v.y;
            x[4 * k + 2] = v.z;
            x[4 * k + 3] = v.w;
        }
        if (part == 3) {                                         // columns 48..63
            x[3] = 0.f;                                          // V
            x[4] = 0.f;                                          // e
            x[5] = a.env.spread;
            x[6] = x[7] = x[8] = 1.f;                            // bias pieces
#pragma unroll
            for (int j = 9; j < 16; ++j) x[j] = 0.f;
        }
        if (!valid) {
#pragma unroll
            for (int j = 0; j < 16; ++j) x[j] = 0.f;
        }
        put_row<true, 16>(X, ei, 16 * part, x);
    };

    const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
    const uint32_t sX = smem_u32(X), sH1 = smem_u32(H1), sH2 = smem_u32(H2), sImg = smem_u32(img);
    issue_rows(0);
    issue_rows(1);
    issue_rows(2);
    int t = 0;
    if (issuer) {
        // the same CTA barriers as the workers, each followed by its MMAs
        ok = __syncthreads_and(ok);
        tc_fence_after();
        if (ok && leader && L > 0) {
            issue_layer<true>(tmem + kD1, sX, sImg + w.actor_off[0], G::XC, kActorH1);
            mma_commit(&bar_l1);
        }
        for (; t < L; ++t) {
            if (!__syncthreads_and(ok)) break;                  // barrier A: H1 of step t
            tc_fence_after();
            if (leader) {
                issue_layer<true>(tmem + kD2, sH1, sImg + w.actor_off[1], G::H1C, kActorH2);
                mma_commit(&bar_mma);
            }
            barrier_b();                                         // H2 of step t, X of step t+1
            tc_fence_after();
            if (leader) {
                issue_layer<true>(tmem + kD3, sH2, sImg + w.actor_off[2], G::H2C, 48);
                mma_commit(&bar_mma);
                if (t + 1 < L) {
                    issue_layer<true>(tmem + kD1, sX, sImg + w.actor_off[0], G::XC, kActorH1);
                    mma_commit(&bar_l1);
                }
            }
        }
    } else if (loader) {
        ok = __syncthreads_and(ok);                              // the workers' first state tile
        for (; t < L; ++t) {
            if (!__syncthreads_and(ok)) break;                  // barrier A of step t
            issue_rows(t + 3);                  // slot (t+3)%3 held step t's rows, last read in step t-1
        }
    } else {
        uint32_t ph = 0, ph1 = 0;
        ok = ok && wait_rows(0);
        build_x(0);
        fence_async_smem();                                          // X and the edited W1 tile, for the MMA
        tc_fence_before();
        ok = __syncthreads_and(ok);
        tc_fence_after();

        int p_act = 0, p_label = 0, p_done = 0;
        float p_pnl = 0.f, p_logp = 0.f, p_vin = 0.f, p_vpost = 0.f;
        bool p_store = false;
        auto flush_out = [&](int t) {
            if (live && part < 3) {
                if (part == 0) {
                    a.actions[row0 + t] = p_store ? p_act : 0;
                    a.logp[row0 + t] = p_store ? p_logp : 0.f;
                } else if (part == 1) {
                    a.dones[row0 + t] = p_store ? p_done : 0;
                    a.v_in[row0 + t] = p_store ? p_vin : 0.f;
                } else {
                    a.v_post[row0 + t] = p_store ? p_vpost : 0.f;
                }
            }
        };
        auto window_reward = [&](int t) {
            const float rew = env_window_reward(st, p_act, p_pnl, p_label, p_done, env);
            if (live) a.rewards[row0 + t] = p_store ? rew : 0.f;
        };

        for (; t < L; ++t) {                       // leaves only at the CTA-uniform test below
            ok = ok && mbar_wait(&bar_l1, ph1, abort) && wait_rows(t + 1);
            ph1 ^= 1;
            tc_fence_after();
            // ---- layer 1 epilogue, columns [32p, +32): + bf16(V) W1[:,51] + e W1[:,52]
            {
                float v[32];
                tmem_ld32(lane_addr + kD1 + 32 * part, v);
                tmem_ld_wait();
                const float2 bv = make_float2(bf16_round(st.V), bf16_round(st.V)), be = make_float2(st.e, st.e);
                const float4 *wv = reinterpret_cast<const float4 *>(s_wv + 32 * part);
                const float4 *we = reinterpret_cast<const float4 *>(s_we + 32 * part);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const float4 a4 = wv[k], b4 = we[k];
                    float2 lo = make_float2(v[4 * k + 0], v[4 * k + 1]), hi = make_float2(v[4 * k + 2], v[4 * k + 3]);
                    lo = fma2(bv, make_float2(a4.x, a4.y), fma2(be, make_float2(b4.x, b4.y), lo));
                    hi = fma2(bv, make_float2(a4.z, a4.w), fma2(be, make_float2(b4.z, b4.w), hi));
                    v[4 * k + 0] = lo.x;
                    v[4 * k + 1] = lo.y;
                    v[4 * k + 2] = hi.x;
                    v[4 * k + 3] = hi.y;
                }
                float *drow = nullptr;
                if constexpr (kDump) drow = live ? a.dump.row(n, t, L) : nullptr;
                put_row_relu<32, kDump>(H1, ei, 32 * part, v, drow ? drow + a.dump.act_off + 32 * part : nullptr);
            }
            fence_async_smem();
            tc_fence_before();
            if (!__syncthreads_and(ok)) break;      // CTA-uniform exit after a failed wait
            tc_fence_after();
            issue_rows(t + 3);                  // tracks the loaders' `issued`
            // ---- while layer 2 runs: the next state tile, the bar's return, the step before's reward
            if (t + 1 < L) build_x(t + 1);
            const float em1 = valid ? ring_row(t + 1)[12].w : 0.f;   // expm1(F[b+1, 0]) of this step's bar b
            ok = ok && mbar_wait(&bar_mma, ph, abort);
            ph ^= 1;
            tc_fence_after();
            // ---- layer 2 epilogue, columns [16p, +16)
            {
                float v[16];
                tmem_ld_x<16>(lane_addr + kD2 + 16 * part, v);
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] += bias[16 * part + j];
                float *drow = nullptr;
                if constexpr (kDump) drow = live ? a.dump.row(n, t, L) : nullptr;
                put_row_relu<16, kDump>(H2, ei, 16 * part, v,
                                        drow ? drow + a.dump.act_off + kActorH1 + 16 * part : nullptr);
            }
            fence_async_smem();
            tc_fence_before();
            barrier_b();
            tc_fence_after();
            if (t > 0) flush_out(t - 1);
            if (part == 3 && t > 0) window_reward(t - 1);
            ok = ok && mbar_wait(&bar_mma, ph, abort);
            ph ^= 1;
            tc_fence_after();
            // ---- logits [12p, +12) (45 valid), block maximum and sum
            const int nv = part < 3 ? kLogitsPerPart : kActions - 3 * kLogitsPerPart;
            float lg[kLogitsPerPart], q[kLogitsPerPart];
#pragma unroll
            for (int i = 0; i < kLogitsPerPart / 4; ++i)
                tmem_ld_x<4>(lane_addr + kD3 + kLogitsPerPart * part + 4 * i, lg + 4 * i);
            tmem_ld_wait();
            const float u = lcg_uniform(st.rng);                     // every part's LCG copy advances alike
            float mp = -INFINITY;
#pragma unroll
            for (int j = 0; j < kLogitsPerPart; ++j) {
                lg[j] += bias[kActorH2 + kLogitsPerPart * part + j];
                if (j < nv) mp = fmaxf(mp, lg[j]);
            }
            float sp = 0.f;
#pragma unroll
            for (int j = 0; j < kLogitsPerPart; ++j) {
                q[j] = j < nv ? __expf(lg[j] - mp) : 0.f;
                sp += q[j];
            }
            s_ms[part][ei] = make_float2(mp, sp);
            qsync(quarter);
            float2 ms[4];
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) ms[pp] = s_ms[pp][ei];
            const float m = fmaxf(fmaxf(ms[0].x, ms[1].x), fmaxf(ms[2].x, ms[3].x));
            float S = 0.f, base = 0.f, scale = 1.f;
#pragma unroll
            for (int pp = 0; pp < 4; ++pp) {
                const float sc = __expf(ms[pp].x - m);
                if (pp == part) {
                    base = S;
                    scale = sc;
                }
                S = fmaf(ms[pp].y, sc, S);
            }
            const float thr = u * S;
            float run = base;
            int cand = kNone;
            float lcand = 0.f;
#pragma unroll
            for (int j = 0; j < kLogitsPerPart; ++j) {
                if (j < nv) {
                    run = fmaf(q[j], scale, run);
                    if (cand == kNone && thr < run) {
                        cand = kLogitsPerPart * part + j;
                        lcand = lg[j];
                    }
                }
            }
            if (part == 3 && cand == kNone) {                        // u*S above every running sum: action 44
                cand = kActions - 1;
                lcand = lg[kActions - 1 - 3 * kLogitsPerPart];
            }
            s_cand[part][ei] = cand;
            s_la[part][ei] = lcand;
            qsync(quarter);
            int act = kActions - 1, pa = 3;
#pragma unroll
            for (int pp = 3; pp >= 0; --pp)
                if (s_cand[pp][ei] != kNone) {
                    act = s_cand[pp][ei];
                    pa = pp;
                }
            // ---- the trade step, in every part
            const float v_in = st.V;
            float pnl, v_post;
            int label, done;
            env_trade(st, act, em1, env, pnl, v_post, label, done);
            const bool store = valid && ok;
            if (part == 0) p_logp = (s_la[pa][ei] - m) - logf(S);
            p_vin = v_in;
            p_vpost = v_post;
            p_act = act;
            p_pnl = pnl;
            p_label = label;
            p_done = done;
            p_store = store;
        }
        if (part == 3 && t == L && L > 0) window_reward(L - 1);
        if (t == L && L > 0) flush_out(L - 1);
    }
    if (worker) {
        if (!ok) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
        // rows still in flight after an early exit land before the CTA ends
        int never = 0;
        for (int s = waited + 1; s <= issued; ++s)
            mbar_wait(&bar_rows[s % 3], (uint32_t)((s / 3) & 1), &never, 100000000ull);
    }
    if (leader) {
        mma_commit(&bar_final);                                  // every MMA completes before TMEM is released
        int never = 0;
        mbar_wait(&bar_final, 0, &never, 100000000ull);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kP1TmemCols);
}

template <bool BF16, bool kDump>
cudaError_t launch_p1(const Phase1Args &a, const UmmaWeights &w, const CUtensorMap &fmap, cudaStream_t s)
{
    using G = P1Geo<BF16>;
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(phase1_umma_kernel<BF16, kDump>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, G::SMEM);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    const int blocks = (a.N + kP1Threads - 1) / kP1Threads;
    phase1_umma_kernel<BF16, kDump><<<blocks, kP1Threads, G::SMEM, s>>>(a, w, fmap);
    return cudaGetLastError();
}

template <bool kDump>
cudaError_t launch_bf16(const Phase1Args &a, const UmmaWeights &w, const CUtensorMap &fmap, cudaStream_t s)
{
    using G = P1Geo<true>;
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(phase1_bf16_kernel<kDump>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 G::SMEM);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    const int blocks = (a.N + kP1Threads - 1) / kP1Threads;
    phase1_bf16_kernel<kDump><<<blocks, kQThreads, G::SMEM, s>>>(a, w, fmap);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_phase1_umma(const Phase1Args &a, const UmmaWeights &w, const CUtensorMap &fmap, cudaStream_t s)
{
    const bool dump = a.dump.p != nullptr;
    if (!w.bf16) return dump ? launch_p1<false, true>(a, w, fmap, s) : launch_p1<false, false>(a, w, fmap, s);
    return dump ? launch_bf16<true>(a, w, fmap, s) : launch_bf16<false>(a, w, fmap, s);
}

namespace {

// the feature matrix with rows padded to kFPad floats (a tensor map's row
// pitch must be a multiple of 16 bytes, 51 floats -- 204 bytes -- is not); the
// extra column carries expm1(F[b, 0]), the bar's simple return, which the
// environment step needs for the bar after its own
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
        if (c0 + 3 == kMarket) v[3] = expm1f(__ldg(F + b * kMarket));   // the bar's simple return
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
