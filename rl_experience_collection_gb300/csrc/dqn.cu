// dqn.cu -- the DQN experience collector (include/dqn.h) on tcgen05 tensor
// cores, bf16 operands, float32 accumulation in TMEM.
//
// Page "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA Experience Collection",
// "Data Flow" (steps 1-15) and "Kernel Components" 1 (dueling Q network), 7
// (TD error), 8 (LCG); the environment is the PPO collector's (env.cuh).
//
// Three stream-ordered phases, as in the PPO collector:
//   rollout (dqn_rollout_kernel): a CTA owns 128 episodes and steps them
//     together.  Per step the online network's four layers run as M = 128
//     MMAs: L1 X[128 x 64] W1^T -> 256, L2 H W2^T -> 256, L3 H [Wv1; Wa1]^T ->
//     256 (value and advantage hidden units side by side), head H Wh^T -> 48
//     (Wh block-diagonal: advantage rows 0..44 read the advantage half, row 45
//     the value half).  The epilogues add the bias, apply LeakyReLU(0.01) and
//     round to bf16 into the next layer's operand; the head's epilogue forms
//     Q = V + (A - mean A), picks the action (epsilon-greedy) and steps the
//     environment.  The weights (312 KB a step) stream from L2 through a
//     three-stage ring of 32 KB bulk copies; activations stay in shared memory.
//   state rows (states.cu).
//   target pass (dqn_target_kernel): every transition at once, in tiles of 128
//     rows: the curiosity model on [x ; one-hot a] against the pre-reset next
//     state x', and the target network on x'; the epilogues add the curiosity
//     bonus to the reward and form the TD error.
// Between the phases out_td holds V entering each step and a handle-owned
// array V' after the trade.
//
// Warp roles (both kernels): warps 0-7 are row warps (warp w serves TMEM lanes
// and rows 32 (w % 4) .. + 31 and the column half w / 4 of each layer), warps
// 8-10 stream the weights, warp 8 + s filling ring stage s (the bulk copies of
// one warp complete one after another, those of different warps overlap), and
// warp 11 allocates TMEM and one lane issues the MMAs.  Every wait is bounded; a wait that gives up sets a flag
// that ends every role's loop, and the status word records the timeout.
#include <math.h>
#include <string.h>

#include <functional>
#include <new>
#include <vector>

#include "../../include/dqn.h"
#include "env.cuh"
#include "umma.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kH = 256, kHeadN = 48;
constexpr int kRowWarps = 8;
constexpr int kStages = 3;
constexpr int kProdWarp0 = 8, kMmaWarp = kProdWarp0 + kStages, kThreads = (kMmaWarp + 1) * 32;
constexpr int kChunk = 128 * 128;                   // one K-chunk (64 bf16 columns) of 128 rows
constexpr int kStage = 32 * 1024;
constexpr int kNetUnits = 10;                       // W1, W2 x4, W3 x4, head
constexpr int kTargetUnits = 11;                    // curiosity C1|C2, then the target net's 10
constexpr int kHeadTile = kHeadN * 128;             // one K-chunk of the head's 48 rows (6 KB)
constexpr int kCurTile = 64 * 128;                  // C1 or C2 (64 rows, 8 KB)
constexpr int kBiasFloats = 3 * kH + kHeadN;        // b1 | b2 | [bv1 ; ba1] | [ba2, bv2, 0, 0]

// ---- weight image (one device allocation), offsets in bytes
struct DqnImage {
    const uint8_t *base = nullptr;
    long long unit_off[kNetUnits + kTargetUnits] = {};   // online units, then the target pass's
    uint32_t unit_bytes[kNetUnits + kTargetUnits] = {};
    const float *online_bias = nullptr, *target_bias = nullptr;   // kBiasFloats each
    const float *cur_b1 = nullptr;       // [64]
    const float *cur_b2 = nullptr;       // [64] (54 valid)
    const float *cur_onehot = nullptr;   // [45][64]: bf16-rounded C1[:, 54 + a]
};

struct RolloutArgs {
    const float *F;
    const int32_t *starts;
    const uint32_t *seeds;
    int N, L, n_bars;
    float epsilon;
    int32_t *actions, *dones;
    float *rewards;      // base reward (the target pass adds the curiosity bonus)
    float *v_in;         // V entering each step (out_td until the target pass)
    float *v_post;       // V' after the trade
    float *q;            // online Q of the action taken
    int *status;
    EnvConst env;
};

struct TargetArgs {
    const float *F;
    const int32_t *starts;
    int N, L, n_bars;
    float gamma;
    const int32_t *actions, *dones;
    float *rewards;      // in: base reward; out: + curiosity bonus
    float *td;           // in: V entering each step; out: TD error
    const float *v_post;
    const float *q;
    float *next_states;  // [N, L, 54] or null
    int *status;
    EnvConst env;
};

__device__ __forceinline__ float leaky(float x) { return x > 0.f ? x : 0.01f * x; }

// 32 consecutive columns [c0, c0 + 32) of row r (c0 a multiple of 32), rounded
// to bf16, into a chunked, 128-byte-swizzled operand buffer
__device__ __forceinline__ void put32(uint8_t *buf, int r, int c0, const float (&v)[32])
{
    uint8_t *chunk = buf + (c0 >> 6) * kChunk;
    const int u0 = (c0 & 63) >> 3;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint4 p;
        p.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
        p.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
        p.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
        p.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
        *reinterpret_cast<uint4 *>(chunk + sw128_offset(r, u0 + q)) = p;
    }
}

// the warp's 32 rows, columns [c0, c0 + 32) of the accumulator at TMEM column
// `col`, + bias, LeakyReLU, into the operand buffer
__device__ __forceinline__ void drain32_leaky(uint32_t taddr, int col, const float *bias, uint8_t *buf, int r,
                                              int c0)
{
    float v[32];
    tmem_ld32(taddr + col, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = leaky(v[i] + bias[c0 + i]);
    put32(buf, r, c0, v);
}

// columns of a state row [F[b, 0..50], V, e, spread, 0 x 10] (or of x'), Frow
// the feature row F[b]: column half 1 holds columns 0..31, half 0 32..63
__device__ __forceinline__ void state_cols(const float *Frow, float V, float e, float spread, int hf, bool valid,
                                           float (&v)[32])
{
    if (hf == 1) {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = valid ? __ldg(Frow + i) : 0.f;
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            const int c = 32 + i;
            float x = 0.f;
            if (valid) {
                if (c < kMarket) x = __ldg(Frow + c);
                else if (c == kMarket) x = V;
                else if (c == kMarket + 1) x = e;
                else if (c == kMarket + 2) x = spread;
            }
            v[i] = x;
        }
    }
}

__device__ __forceinline__ int state_c0(int hf) { return hf == 1 ? 0 : 32; }

// a row warp's wait: every lane waits, and the warp goes on only if all of them
// saw the phase, so that the warp-wide TMEM loads after it are never reached by
// part of a warp (a lane can give up at the moment another sees the phase)
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    return __all_sync(0xffffffffu, mbar_wait(bar, parity, abort));
}

// waits with a time limit only (the drain at exit, after a give-up)
__device__ __forceinline__ void mbar_wait_drain(uint64_t *bar, uint32_t parity)
{
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > 1000000000ull) return;
}

// one layer's MMAs: A = nk K-chunks at `a` (chunk stride kChunk), B = the
// stage's tiles (chunk stride b_stride), N columns into TMEM column d
__device__ __forceinline__ void mma_layer(uint32_t d, const uint8_t *a, const uint8_t *b, int b_stride, int nk,
                                          uint32_t id, bool accumulate_first)
{
    for (int c = 0; c < nk; ++c)
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma<true>(d, desc_sw128(smem_u32(a + c * kChunk + 32 * k)), desc_sw128(smem_u32(b + c * b_stride + 32 * k)),
                      id, (accumulate_first || c > 0 || k > 0) ? 1u : 0u);
}

// ---------------------------------------------------------------------------
// rollout: the online network inside the serial step loop

struct RBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t x_ready;     // rows -> MMA: the step's state rows are in X (8 warp arrivals)
    uint64_t h_ready;     // rows -> MMA: a hidden layer is in H (8 warp arrivals, 3 a step)
    uint64_t acc;         // MMA -> rows: a layer's accumulator is complete (4 a step)
    uint64_t fin;         // MMA: everything issued has completed (exit)
};

constexpr int kRSmem = 1024 + kChunk + 4 * kChunk + kStages * kStage + kBiasFloats * 4 + 1024;
static_assert(kRSmem <= 232448, "rollout shared memory");

__global__ void __launch_bounds__(kThreads, 1) dqn_rollout_kernel(RolloutArgs a, DqnImage w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *X = base;                          // 1 K-chunk
    uint8_t *Hb = X + kChunk;                   // 4 K-chunks
    uint8_t *ring = Hb + 4 * kChunk;
    float *bias = reinterpret_cast<float *>(ring + kStages * kStage);
    RBars *bars = reinterpret_cast<RBars *>(bias + kBiasFloats);
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;
    __shared__ uint32_t div_s[kDivWords];

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->x_ready, kRowWarps);
        mbar_init(&bars->h_ready, kRowWarps);
        mbar_init(&bars->acc, 1);
        mbar_init(&bars->fin, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < kBiasFloats; i += kThreads) bias[i] = w.online_bias[i];
    for (int i = tid; i < kDivWords; i += kThreads) div_s[i] = a.env.div_low[i];
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_s, 256);
        tmem_relinquish();            // this CTA allocates once; later CTAs on the SM may allocate
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    EnvConst env = a.env;
    env.div_low = div_s;
    const int L = a.L;

    if (warp < kRowWarps) {
        // ------------------------------------------------------------ rows
        const int quad = warp & 3, hf = warp >> 2, r = quad * 32 + lane;
        const int n = blockIdx.x * 128 + r;
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
        int start = 0;
        bool valid = n < a.N;
        if (valid) {
            start = a.starts[n];
            if (!start_ok(start, L, a.n_bars)) {
                valid = false;
                if (hf == 0) set_status(a.status, ROLLOUT_ERR_RANGE);
            }
        }
        EpState s;
        ep_reset(s);
        s.rng = n < a.N ? a.seeds[n] : 0u;
        uint32_t acc_phase = 0;
        for (int t = 0; t < L; ++t) {
            const long long b = (long long)start + t;
            const float *Frow = a.F + b * kMarket;
            {
                float v[32];
                state_cols(Frow, s.V, s.e, env.spread, hf, valid, v);
                put32(X, r, state_c0(hf), v);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->x_ready);
            // three hidden layers: accumulator -> bias, LeakyReLU, bf16 -> H
            bool ok = true;
            for (int l = 0; l < 3 && ok; ++l) {
                if (!warp_wait(&bars->acc, acc_phase & 1, &abort_flag)) { ok = false; break; }
                ++acc_phase;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int c0 = hf * 128 + 32 * j;
                    drain32_leaky(taddr, c0, bias + l * kH, Hb, r, c0);
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->h_ready);
            }
            if (!ok || !warp_wait(&bars->acc, acc_phase & 1, &abort_flag)) break;
            ++acc_phase;
            tc_fence_after();
            if (hf == 0) {
                // head: A = cols 0..44, V = col 45; Q = V + (A - mean A)
                float d0[32], d1[32];
                tmem_ld32(taddr + 0, d0);
                tmem_ld32(taddr + 32, d1);
                tmem_ld_wait();
                const float *bh = bias + 3 * kH;
                float qv[kActions];
                float sumA = 0.f;
#pragma unroll
                for (int j = 0; j < kActions; ++j) {
                    qv[j] = (j < 32 ? d0[j] : d1[j - 32]) + bh[j];
                    sumA += qv[j];
                }
                const float V = d1[kActions - 32] + bh[kActions];
                const float meanA = sumA / (float)kActions;
                int best = 0;
                float qbest = -INFINITY;
#pragma unroll
                for (int j = 0; j < kActions; ++j) {
                    qv[j] = V + (qv[j] - meanA);
                    if (qv[j] > qbest) { qbest = qv[j]; best = j; }
                }
                // epsilon-greedy: u1 decides, the second state gives the random action
                const float u1 = lcg_uniform(s.rng);
                s.rng = s.rng * 1664525u + 1013904223u;
                const int a_rand = (int)(((uint64_t)(s.rng >> 8) * (uint64_t)kActions) >> 24);
                const int act = (u1 < a.epsilon) ? a_rand : best;
                float q_sel = qv[0];
#pragma unroll
                for (int j = 1; j < kActions; ++j)
                    if (j == act) q_sel = qv[j];
                const long long i = (long long)n * L + t;
                if (valid) {
                    const float v_in = s.V;
                    float pnl, v_post;
                    int label, done;
                    env_trade(s, act, expm1f(__ldg(a.F + (b + 1) * kMarket)), env, pnl, v_post, label, done);
                    const float rew = env_window_reward(s, act, pnl, label, done, env);
                    a.actions[i] = act;
                    a.dones[i] = done;
                    a.rewards[i] = rew;
                    a.v_in[i] = v_in;
                    a.v_post[i] = v_post;
                    a.q[i] = q_sel;
                } else if (n < a.N) {
                    a.actions[i] = 0;
                    a.dones[i] = 0;
                    a.rewards[i] = 0.f;
                    a.v_in[i] = 0.f;
                    a.v_post[i] = 0.f;
                    a.q[i] = 0.f;
                }
            }
            tc_fence_before();
        }
    } else if (warp < kMmaWarp) {
        // ------------------------------------------------------------ weight stream, stage st
        const int st = warp - kProdWarp0;
        if (lane == 0) {
            const long long total = (long long)kNetUnits * L;
            long long last = -1;
            for (long long u = st; u < total; u += kStages) {
                const int i = (int)(u % kNetUnits);
                if (u >= kStages && !mbar_wait(&bars->empty[st], (uint32_t)((u / kStages - 1) & 1), &abort_flag))
                    break;
                mbar_arrive_expect_tx(&bars->full[st], w.unit_bytes[i]);
                bulk_g2s(ring + st * kStage, w.base + w.unit_off[i], w.unit_bytes[i], &bars->full[st]);
                last = u;
            }
            // its last copy completes before the CTA may exit
            if (last >= 0) mbar_wait_drain(&bars->full[st], (uint32_t)((last / kStages) & 1));
        }
    } else {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t id256 = idesc(true, 128, kH), id48 = idesc(true, 128, kHeadN);
            long long u = 0;
            uint32_t h_phase = 0;
            bool ok = true;
            for (int t = 0; t < L && ok; ++t) {
                if (!mbar_wait(&bars->x_ready, (uint32_t)(t & 1), &abort_flag)) break;
                tc_fence_after();
                for (int layer = 0; layer < 4 && ok; ++layer) {
                    if (layer > 0) {
                        if (!mbar_wait(&bars->h_ready, h_phase & 1, &abort_flag)) { ok = false; break; }
                        ++h_phase;
                        tc_fence_after();
                    }
                    const int n_units = (layer == 0 || layer == 3) ? 1 : 4;
                    for (int cu = 0; cu < n_units; ++cu, ++u) {
                        const int st = (int)(u % kStages);
                        if (!mbar_wait(&bars->full[st], (uint32_t)((u / kStages) & 1), &abort_flag)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint8_t *bsrc = ring + st * kStage;
                        if (layer == 0) mma_layer(tmem, X, bsrc, 0, 1, id256, false);
                        else if (layer == 3) mma_layer(tmem, Hb, bsrc, kHeadTile, 4, id48, false);
                        else mma_layer(tmem, Hb + cu * kChunk, bsrc, 0, 1, id256, cu > 0);
                        mma_commit(&bars->empty[st]);
                    }
                    if (ok) mma_commit(&bars->acc);
                }
            }
            // every MMA issued has completed before TMEM is freed
            mma_commit(&bars->fin);
            mbar_wait_drain(&bars->fin, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
    if (tid == 0 && abort_flag) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
}

// ---------------------------------------------------------------------------
// target pass: curiosity and the target network over every transition

struct TBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t x_ready;     // rows -> MMA: X and X' of the tile are written (8 warp arrivals)
    uint64_t z_ready;     // rows -> MMA: the curiosity hidden layer Z is written
    uint64_t h_ready;     // rows -> MMA: a hidden layer of the target net is in H (3 a tile)
    uint64_t acc_c;       // MMA -> rows: curiosity layer 1, then 2 (2 a tile)
    uint64_t acc_q;       // MMA -> rows: target layers 1..3 and the head (4 a tile)
    uint64_t mse_ready;   // column half 1 -> half 0: its share of the curiosity error (4 warp arrivals)
    uint64_t fin;
};

constexpr int kTSmem = 1024 + 3 * kChunk + 4 * kChunk + kStages * kStage + (kBiasFloats + 128 + 128) * 4 + 1024;
static_assert(kTSmem <= 232448 - 2048, "target pass shared memory");
constexpr uint32_t kTmemQ = 0, kTmemC1 = 256, kTmemC2 = 320;

// kStall: a test build in which the first producer of CTA 0 issues no copy, so
// that CTA's MMA issuer waits on a weight stage that never fills and the
// bounded-wait exit runs (dqn_test_stall)
template <bool kStall>
__global__ void __launch_bounds__(kThreads, 1) dqn_target_kernel(TargetArgs a, DqnImage w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *X = base, *Xn = X + kChunk, *Z = Xn + kChunk;
    uint8_t *Hb = Z + kChunk;
    uint8_t *ring = Hb + 4 * kChunk;
    float *bias = reinterpret_cast<float *>(ring + kStages * kStage);
    float *cb1 = bias + kBiasFloats, *cb2 = cb1 + 64;
    float *mse_part = cb2 + 64;
    TBars *bars = reinterpret_cast<TBars *>(mse_part + 128);
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->x_ready, kRowWarps);
        mbar_init(&bars->z_ready, kRowWarps);
        mbar_init(&bars->h_ready, kRowWarps);
        mbar_init(&bars->acc_c, 1);
        mbar_init(&bars->acc_q, 1);
        mbar_init(&bars->mse_ready, kRowWarps / 2);
        mbar_init(&bars->fin, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < kBiasFloats; i += kThreads) bias[i] = w.target_bias[i];
    for (int i = tid; i < 64; i += kThreads) {
        cb1[i] = w.cur_b1[i];
        cb2[i] = w.cur_b2[i];
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_s, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const long long R = (long long)a.N * a.L;
    const long long n_tiles = (R + 127) / 128;

    if (warp < kRowWarps) {
        // ------------------------------------------------------------ rows
        const int quad = warp & 3, hf = warp >> 2, r = quad * 32 + lane;
        const int c0 = state_c0(hf);
        const uint32_t taddr = tmem + ((uint32_t)(quad * 32) << 16);
        uint32_t pc = 0, pq = 0, it = 0;
        bool ok = true;
        for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
            const long long i = tile * 128 + r;
            bool valid = i < R;
            int act = 0, done = 0;
            float r0 = 0.f, qs = 0.f, vin = 0.f, vp = 0.f, e_in = 0.f;
            long long b = 0;
            if (valid) {
                const long long n = i / a.L;
                const int t = (int)(i - n * a.L);
                const int start = __ldg(a.starts + n);
                valid = start_ok(start, a.L, a.n_bars);
                if (valid) {
                    b = (long long)start + t;
                    act = a.actions[i];
                    // the one-hot row read below stays in bounds whatever the
                    // rollout left here (its rows after a give-up are unwritten)
                    if ((unsigned)act >= (unsigned)kActions) act = 0;
                    done = a.dones[i];
                    r0 = a.rewards[i];
                    qs = a.q[i];
                    vin = a.td[i];
                    vp = a.v_post[i];
                    e_in = (t == 0 || a.dones[i - 1]) ? 0.f : exposure_of(a.actions[i - 1]);
                }
            }
            float xn[32];
            {
                float v[32];
                state_cols(a.F + b * kMarket, vin, e_in, a.env.spread, hf, valid, v);
                put32(X, r, c0, v);
                state_cols(a.F + (b + 1) * kMarket, vp, exposure_of(act), a.env.spread, hf, valid, xn);
                put32(Xn, r, c0, xn);
            }
            fence_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->x_ready);
            // curiosity layer 1: Z = ReLU(X C1^T + c1 + C1[:, 54 + a])
            if (!warp_wait(&bars->acc_c, pc & 1, &abort_flag)) break;
            ++pc;
            tc_fence_after();
            {
                float v[32];
                tmem_ld32(taddr + kTmemC1 + c0, v);
                tmem_ld_wait();
                const float *oh = w.cur_onehot + act * 64 + c0;
#pragma unroll
                for (int k = 0; k < 32; ++k) v[k] = relu(v[k] + cb1[c0 + k] + __ldg(oh + k));
                put32(Z, r, c0, v);
            }
            fence_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->z_ready);
            // target layer 1, then curiosity layer 2, then target layers 2, 3
            float cur = 0.f;
            for (int l = 0; l < 3 && ok; ++l) {
                if (!warp_wait(&bars->acc_q, pq & 1, &abort_flag)) { ok = false; break; }
                ++pq;
                tc_fence_after();
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int cc = hf * 128 + 32 * j;
                    drain32_leaky(taddr + kTmemQ, cc, bias + l * kH, Hb, r, cc);
                }
                fence_async_smem();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->h_ready);
                if (l == 0) {
                    // curiosity layer 2: squared error against x' over the 54 state columns
                    if (!warp_wait(&bars->acc_c, pc & 1, &abort_flag)) { ok = false; break; }
                    ++pc;
                    tc_fence_after();
                    float v[32];
                    tmem_ld32(taddr + kTmemC2 + c0, v);
                    tmem_ld_wait();
                    float part = 0.f;
#pragma unroll
                    for (int k = 0; k < 32; ++k)
                        if (c0 + k < kState) {
                            const float dlt = (v[k] + cb2[c0 + k]) - xn[k];
                            part += dlt * dlt;
                        }
                    tc_fence_before();
                    if (hf == 1) {
                        mse_part[r] = part;
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&bars->mse_ready);
                    } else {
                        if (!warp_wait(&bars->mse_ready, it & 1, &abort_flag)) { ok = false; break; }
                        cur = a.env.cur_coef * ((mse_part[r] + part) / (float)kState);
                    }
                }
            }
            if (!ok || !warp_wait(&bars->acc_q, pq & 1, &abort_flag)) break;
            ++pq;
            tc_fence_after();
            if (hf == 0) {
                // the TMEM loads are warp-wide (.sync.aligned): every lane of the
                // warp issues them, rows past the end included; only stores are per row
                float d0[32], d1[32];
                tmem_ld32(taddr + kTmemQ, d0);
                tmem_ld32(taddr + kTmemQ + 32, d1);
                tmem_ld_wait();
                const float *bh = bias + 3 * kH;
                float sumA = 0.f;
#pragma unroll
                for (int j = 0; j < kActions; ++j) sumA += (j < 32 ? d0[j] : d1[j - 32]) + bh[j];
                const float V = d1[kActions - 32] + bh[kActions];
                const float meanA = sumA / (float)kActions;
                float qmax = -INFINITY;
#pragma unroll
                for (int j = 0; j < kActions; ++j) qmax = fmaxf(qmax, V + (((j < 32 ? d0[j] : d1[j - 32]) + bh[j]) - meanA));
                if (valid) {
                    const float rew = r0 + cur;
                    a.rewards[i] = rew;
                    a.td[i] = fabsf(rew + a.gamma * qmax * (1.f - (float)done) - qs);
                } else if (i < R) {
                    a.rewards[i] = 0.f;
                    a.td[i] = 0.f;
                }
            }
            if (a.next_states && i < R) {
                float *dst = a.next_states + i * kState + c0;
#pragma unroll
                for (int k = 0; k < 32; ++k)
                    if (c0 + k < kState) dst[k] = valid ? xn[k] : 0.f;
            }
            tc_fence_before();
        }
    } else if (warp < kMmaWarp) {
        const int st = warp - kProdWarp0;
        if (lane == 0) {
            const long long my_tiles = n_tiles > blockIdx.x ? (n_tiles - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
            const long long total = (kStall && blockIdx.x == 0 && st == 0) ? 0 : my_tiles * kTargetUnits;
            long long last = -1;
            for (long long u = st; u < total; u += kStages) {
                const int i = kNetUnits + (int)(u % kTargetUnits);
                if (u >= kStages && !mbar_wait(&bars->empty[st], (uint32_t)((u / kStages - 1) & 1), &abort_flag))
                    break;
                mbar_arrive_expect_tx(&bars->full[st], w.unit_bytes[i]);
                bulk_g2s(ring + st * kStage, w.base + w.unit_off[i], w.unit_bytes[i], &bars->full[st]);
                last = u;
            }
            if (last >= 0) mbar_wait_drain(&bars->full[st], (uint32_t)((last / kStages) & 1));
        }
    } else {
        if (lane == 0) {
            const uint32_t id256 = idesc(true, 128, kH), id48 = idesc(true, 128, kHeadN), id64 = idesc(true, 128, 64);
            long long u = 0;
            uint32_t it = 0, hp = 0;
            bool ok = true;
            auto take = [&](long long unit, int &st) -> bool {
                st = (int)(unit % kStages);
                if (!mbar_wait(&bars->full[st], (uint32_t)((unit / kStages) & 1), &abort_flag)) return false;
                tc_fence_after();
                return true;
            };
            for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
                if (!mbar_wait(&bars->x_ready, it & 1, &abort_flag)) break;
                tc_fence_after();
                int s_cur, st;
                // curiosity layer 1 (its unit's second tile, C2, waits for Z)
                if (!take(u, s_cur)) break;
                ++u;
                mma_layer(tmem + kTmemC1, X, ring + s_cur * kStage, 0, 1, id64, false);
                mma_commit(&bars->acc_c);
                // target layer 1 on X'
                if (!take(u, st)) break;
                ++u;
                mma_layer(tmem + kTmemQ, Xn, ring + st * kStage, 0, 1, id256, false);
                mma_commit(&bars->empty[st]);
                mma_commit(&bars->acc_q);
                // curiosity layer 2
                if (!mbar_wait(&bars->z_ready, it & 1, &abort_flag)) break;
                tc_fence_after();
                mma_layer(tmem + kTmemC2, Z, ring + s_cur * kStage + kCurTile, 0, 1, id64, false);
                mma_commit(&bars->empty[s_cur]);
                mma_commit(&bars->acc_c);
                // target layers 2, 3 (4 units each) and the head
                for (int layer = 1; layer < 4 && ok; ++layer) {
                    if (!mbar_wait(&bars->h_ready, hp & 1, &abort_flag)) { ok = false; break; }
                    ++hp;
                    tc_fence_after();
                    const int n_units = layer == 3 ? 1 : 4;
                    for (int cu = 0; cu < n_units; ++cu) {
                        if (!take(u, st)) { ok = false; break; }
                        ++u;
                        if (layer == 3) mma_layer(tmem + kTmemQ, Hb, ring + st * kStage, kHeadTile, 4, id48, false);
                        else mma_layer(tmem + kTmemQ, Hb + cu * kChunk, ring + st * kStage, 0, 1, id256, cu > 0);
                        mma_commit(&bars->empty[st]);
                    }
                    if (ok) mma_commit(&bars->acc_q);
                }
            }
            mma_commit(&bars->fin);
            mbar_wait_drain(&bars->fin, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && abort_flag) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
}

}  // namespace
}  // namespace rl

// ---------------------------------------------------------------------------
// host: weight conversion and the C ABI

struct dqn_handle {
    rollout_dims dims{};
    int device = 0, sms = 0;
    void *d_img = nullptr;
    size_t img_bytes = 0;
    rl::DqnImage img;
    uint32_t *d_div = nullptr;
    int *d_status = nullptr;
    float *d_vpost = nullptr;
    size_t vpost_cap = 0;
    cudaStream_t last_stream = nullptr;
    bool timing = false, timed_run = false;
    cudaEvent_t ev[4] = {};
    bool test_stall = false;   // dqn_test_stall: launch the target pass's stalling test build
};

namespace rl {
namespace {

// one net's float offsets in the packed host buffer
struct NetLayout {
    size_t w1, b1, w2, b2, wv1, bv1, wv2, bv2, wa1, ba1, wa2, ba2, total;
};

NetLayout net_layout()
{
    NetLayout lo{};
    size_t off = 0;
    lo.w1 = off; off += (size_t)kH * kState;
    lo.b1 = off; off += kH;
    lo.w2 = off; off += (size_t)kH * kH;
    lo.b2 = off; off += kH;
    lo.wv1 = off; off += (size_t)128 * kH;
    lo.bv1 = off; off += 128;
    lo.wv2 = off; off += 128;
    lo.bv2 = off; off += 1;
    lo.wa1 = off; off += (size_t)128 * kH;
    lo.ba1 = off; off += 128;
    lo.wa2 = off; off += (size_t)kActions * 128;
    lo.ba2 = off; off += kActions;
    lo.total = off;
    return lo;
}

constexpr size_t kCurFloats = (size_t)kCurH * (kState + kActions) + kCurH + (size_t)kState * kCurH + kState;

uint16_t bf16_bits(float x)
{
    uint32_t u;
    memcpy(&u, &x, 4);
    return (uint16_t)((u + 0x7FFFu + ((u >> 16) & 1u)) >> 16);     // nearest even (finite inputs)
}

float bf16_value(float x)
{
    const uint32_t u = (uint32_t)bf16_bits(x) << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

// rows [row0, row0 + nrows) of W[n_out][ld] (columns [0, k_valid), K-chunk
// `chunk` of 64), bf16, as a K-major 128-byte-swizzled tile (the layout of
// umma.cuh), appended to out; zero outside the matrix
void put_tile(std::vector<uint8_t> &out, const float *W, int n_out, int ld, int k_valid, int row0, int nrows,
              int chunk)
{
    const size_t base = out.size();
    out.resize(base + (size_t)nrows * 128, 0);
    for (int r = 0; r < nrows; ++r) {
        const int n = row0 + r;
        for (int c = 0; c < 64; ++c) {
            const int k = chunk * 64 + c;
            const float v = (n < n_out && k < k_valid) ? W[(size_t)n * ld + k] : 0.f;
            const int byte = c * 2, unit = byte >> 4, within = byte & 15;
            const size_t off = base + (size_t)(r >> 3) * 1024 + (r & 7) * 128 + ((unit ^ (r & 7)) << 4) + within;
            const uint16_t b = bf16_bits(v);
            memcpy(&out[off], &b, 2);
        }
    }
}

// one net: its ten units appended to img (offsets recorded from unit index u0) and its bias vector
void pack_net(const float *net, std::vector<uint8_t> &img, long long *off, uint32_t *bytes, std::vector<float> &bias)
{
    const NetLayout lo = net_layout();
    auto unit = [&](int i, const std::function<void()> &emit) {
        off[i] = (long long)img.size();
        emit();
        bytes[i] = (uint32_t)((long long)img.size() - off[i]);
    };
    unit(0, [&] { put_tile(img, net + lo.w1, kH, kState, kState, 0, kH, 0); });
    for (int c = 0; c < 4; ++c) unit(1 + c, [&] { put_tile(img, net + lo.w2, kH, kH, kH, 0, kH, c); });
    std::vector<float> w3((size_t)kH * kH);
    memcpy(w3.data(), net + lo.wv1, sizeof(float) * 128 * kH);
    memcpy(w3.data() + 128 * kH, net + lo.wa1, sizeof(float) * 128 * kH);
    for (int c = 0; c < 4; ++c) unit(5 + c, [&] { put_tile(img, w3.data(), kH, kH, kH, 0, kH, c); });
    std::vector<float> wh((size_t)kHeadN * kH, 0.f);
    for (int j = 0; j < kActions; ++j)
        for (int i = 0; i < 128; ++i) wh[(size_t)j * kH + 128 + i] = net[lo.wa2 + (size_t)j * 128 + i];
    for (int i = 0; i < 128; ++i) wh[(size_t)kActions * kH + i] = net[lo.wv2 + i];
    unit(9, [&] {
        for (int c = 0; c < 4; ++c) put_tile(img, wh.data(), kHeadN, kH, kH, 0, kHeadN, c);
    });
    bias.assign(kBiasFloats, 0.f);
    memcpy(&bias[0], net + lo.b1, sizeof(float) * kH);
    memcpy(&bias[kH], net + lo.b2, sizeof(float) * kH);
    memcpy(&bias[2 * kH], net + lo.bv1, sizeof(float) * 128);
    memcpy(&bias[2 * kH + 128], net + lo.ba1, sizeof(float) * 128);
    memcpy(&bias[3 * kH], net + lo.ba2, sizeof(float) * kActions);
    bias[3 * kH + kActions] = net[lo.bv2];
}

int cuda_fail(cudaError_t e, const char *what)
{
    return set_error(e == cudaErrorMemoryAllocation ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA, "%s: %s", what,
                     cudaGetErrorString(e));
}

int upload(dqn_handle *h, const float *weights)
{
    const NetLayout lo = net_layout();
    const size_t total = 2 * lo.total + kCurFloats;
    for (size_t i = 0; i < total; ++i)
        if (!isfinite(weights[i])) return set_error(ROLLOUT_ERR_INVALID, "weight %zu is not finite", i);
    std::vector<uint8_t> img;
    DqnImage &m = h->img;
    std::vector<float> ob, tb;
    pack_net(weights, img, m.unit_off, m.unit_bytes, ob);
    // the target pass: curiosity unit [C1 | C2], then the target net
    const float *cw = weights + 2 * lo.total;
    const float *C1 = cw, *c1 = C1 + (size_t)kCurH * (kState + kActions), *C2 = c1 + kCurH, *c2 = C2 + (size_t)kState * kCurH;
    m.unit_off[kNetUnits] = (long long)img.size();
    put_tile(img, C1, kCurH, kState + kActions, kState, 0, 64, 0);
    put_tile(img, C2, kState, kCurH, kCurH, 0, 64, 0);
    m.unit_bytes[kNetUnits] = (uint32_t)((long long)img.size() - m.unit_off[kNetUnits]);
    pack_net(weights + lo.total, img, m.unit_off + kNetUnits + 1, m.unit_bytes + kNetUnits + 1, tb);
    std::vector<float> vec;
    vec.insert(vec.end(), ob.begin(), ob.end());
    vec.insert(vec.end(), tb.begin(), tb.end());
    vec.insert(vec.end(), c1, c1 + kCurH);
    for (int j = 0; j < 64; ++j) vec.push_back(j < kState ? c2[j] : 0.f);
    for (int a = 0; a < kActions; ++a)
        for (int j = 0; j < kCurH; ++j) vec.push_back(bf16_value(C1[(size_t)j * (kState + kActions) + kState + a]));
    const size_t vec_off = (img.size() + 1023) & ~(size_t)1023;
    const size_t bytes = vec_off + vec.size() * 4;
    std::vector<uint8_t> all(bytes, 0);
    memcpy(all.data(), img.data(), img.size());
    memcpy(all.data() + vec_off, vec.data(), vec.size() * 4);
    cudaError_t e;
    if (h->d_img && h->img_bytes != bytes) {
        cudaFree(h->d_img);
        h->d_img = nullptr;
    }
    if (!h->d_img) {
        if ((e = cudaMalloc(&h->d_img, bytes)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(weights)");
        h->img_bytes = bytes;
    }
    if ((e = cudaMemcpy(h->d_img, all.data(), bytes, cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(weights)");
    const uint8_t *dev = static_cast<const uint8_t *>(h->d_img);
    const float *dv = reinterpret_cast<const float *>(dev + vec_off);
    m.base = dev;
    m.online_bias = dv;
    m.target_bias = dv + kBiasFloats;
    m.cur_b1 = dv + 2 * kBiasFloats;
    m.cur_b2 = m.cur_b1 + 64;
    m.cur_onehot = m.cur_b2 + 64;
    return ROLLOUT_OK;
}

// the diversity decision per category histogram, decided in double on the host
// (the same table the PPO collector builds)
int upload_div_table(dqn_handle *h)
{
    std::vector<uint32_t> bits(kDivWords, 0u);
    for (int c0 = 0; c0 < 32; ++c0)
        for (int c1 = 0; c1 < 32; ++c1)
            for (int c2 = 0; c2 < 32; ++c2) {
                const int n = c0 + c1 + c2;
                if (n == 0 || n > h->dims.div_window) continue;
                double H = 0.0;
                const int c[3] = {c0, c1, c2};
                for (int k = 0; k < 3; ++k)
                    if (c[k] > 0) {
                        const double p = (double)c[k] / (double)n;
                        H -= p * log2(p);
                    }
                if (H < (double)h->dims.div_thresh) {
                    const int bit = c0 * 1024 + c1 * 32 + c2;
                    bits[bit >> 5] |= 1u << (bit & 31);
                }
            }
    cudaError_t e;
    if ((e = cudaMalloc(&h->d_div, bits.size() * 4)) != cudaSuccess) return cuda_fail(e, "cudaMalloc(div table)");
    if ((e = cudaMemcpy(h->d_div, bits.data(), bits.size() * 4, cudaMemcpyHostToDevice)) != cudaSuccess)
        return cuda_fail(e, "cudaMemcpy(div table)");
    return ROLLOUT_OK;
}

int check_dims(const rollout_dims *d)
{
    if (d->n_market != kMarket || d->n_actions != kActions || d->cur_h != kCurH)
        return set_error(ROLLOUT_ERR_UNSUPPORTED, "need 51 market features, 45 actions, curiosity 64");
    if (d->dtype != ROLLOUT_BF16) return set_error(ROLLOUT_ERR_UNSUPPORTED, "the DQN collector runs bf16 only");
    if (d->n_bars < 2) return set_error(ROLLOUT_ERR_INVALID, "n_bars must be >= 2");
    if (d->div_window < 1 || d->div_window > 31) return set_error(ROLLOUT_ERR_UNSUPPORTED, "div_window must be in [1, 31]");
    if (d->max_hold < 1) return set_error(ROLLOUT_ERR_INVALID, "max_hold must be >= 1");
    const float fs[] = {d->barrier, d->pt_scale, d->sl_scale, d->div_thresh, d->div_penalty, d->cur_coef,
                        d->risk_coef, d->tx_base, d->spread};
    for (float f : fs)
        if (!isfinite(f)) return set_error(ROLLOUT_ERR_INVALID, "environment constants must be finite");
    return ROLLOUT_OK;
}

void free_handle(dqn_handle *h)
{
    if (!h) return;
    cudaFree(h->d_img);
    cudaFree(h->d_div);
    cudaFree(h->d_status);
    cudaFree(h->d_vpost);
    for (cudaEvent_t e : h->ev)
        if (e) cudaEventDestroy(e);
    delete h;
}

}  // namespace
}  // namespace rl

using namespace rl;

extern "C" {

long long dqn_weight_count(void) { return (long long)(2 * net_layout().total + kCurFloats); }

int dqn_create(const float *weights, const rollout_dims *dims, dqn_handle **out)
{
    clear_error();
    if (!weights || !dims || !out) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    int rc = check_dims(dims);
    if (rc) return rc;
    dqn_handle *h = new (std::nothrow) dqn_handle();
    if (!h) return set_error(ROLLOUT_ERR_NOMEM, "host allocation failed");
    h->dims = *dims;
    cudaError_t e;
    if ((e = cudaGetDevice(&h->device)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device)) != cudaSuccess ||
        (e = cudaMalloc(&h->d_status, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(h->d_status, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_rollout_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_target_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_target_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem)) !=
            cudaSuccess) {
        free_handle(h);
        return cuda_fail(e, "DQN handle setup");
    }
    if ((rc = upload_div_table(h)) || (rc = upload(h, weights))) {
        free_handle(h);
        return rc;
    }
    *out = h;
    return ROLLOUT_OK;
}

int dqn_set_weights(dqn_handle *h, const float *weights)
{
    clear_error();
    if (!h || !weights) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
    return upload(h, weights);
}

int dqn_run(dqn_handle *h, const float *features, const int32_t *starts, const uint32_t *seeds, int N, int L,
            float gamma, float epsilon, float *states, int32_t *actions, float *rewards, int32_t *dones, float *q,
            float *td, float *next_states, void *stream)
{
    clear_error();
    if (!h || !features || !starts || !seeds || !states || !actions || !rewards || !dones || !q || !td)
        return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (N < 1 || L < 1) return set_error(ROLLOUT_ERR_INVALID, "N and L must be >= 1");
    if (L > h->dims.n_bars - 1) return set_error(ROLLOUT_ERR_INVALID, "L must be <= n_bars - 1");
    if (!isfinite(gamma)) return set_error(ROLLOUT_ERR_INVALID, "gamma must be finite");
    if (!(epsilon >= 0.f && epsilon <= 1.f)) return set_error(ROLLOUT_ERR_INVALID, "epsilon must be in [0, 1]");
    const size_t NL = (size_t)N * (size_t)L;
    cudaError_t e;
    if (NL > h->vpost_cap) {
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(h->d_vpost);
        h->d_vpost = nullptr;
        h->vpost_cap = 0;
        if ((e = cudaMalloc(&h->d_vpost, NL * sizeof(float))) != cudaSuccess) return cuda_fail(e, "cudaMalloc(scratch)");
        h->vpost_cap = NL;
    }
    cudaStream_t s = (cudaStream_t)stream;
    h->last_stream = s;
    const rollout_dims &d = h->dims;
    if ((e = cudaMemsetAsync(h->d_status, 0, sizeof(int), s)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    const EnvConst env{d.barrier, d.max_hold, d.pt_scale, d.sl_scale, d.div_window, d.div_thresh, d.div_penalty,
                       d.cur_coef, d.risk_coef, d.tx_base, d.spread, h->d_div};
    const RolloutArgs ra{features, starts, seeds, N, L, d.n_bars, epsilon, actions, dones, rewards, td, h->d_vpost, q,
                         h->d_status, env};
    auto mark = [&](int i) { return h->timing ? cudaEventRecord(h->ev[i], s) : cudaSuccess; };
    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    dqn_rollout_kernel<<<(N + 127) / 128, kThreads, kRSmem, s>>>(ra, h->img);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "DQN rollout launch");
    if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    const StatesArgs sa{features, starts, N, L, d.n_bars, actions, dones, td, d.spread, states};
    if ((e = launch_states(sa, s)) != cudaSuccess) return cuda_fail(e, "state-row launch");
    if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    const TargetArgs ta{features, starts, N, L, d.n_bars, gamma, actions, dones, rewards, td, h->d_vpost, q,
                        next_states, h->d_status, env};
    const long long tiles = (long long)((NL + 127) / 128);
    const int grid = (int)(tiles < h->sms ? tiles : h->sms);
    if (h->test_stall) dqn_target_kernel<true><<<grid, kThreads, kTSmem, s>>>(ta, h->img);
    else dqn_target_kernel<false><<<grid, kThreads, kTSmem, s>>>(ta, h->img);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "DQN target launch");
    if ((e = mark(3)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    h->timed_run = h->timing;
    return ROLLOUT_OK;
}

int dqn_set_timing(dqn_handle *h, int on)
{
    clear_error();
    if (!h) return set_error(ROLLOUT_ERR_INVALID, "null handle");
    if (on && !h->ev[0])
        for (cudaEvent_t &ev : h->ev) {
            const cudaError_t e = cudaEventCreate(&ev);
            if (e != cudaSuccess) return cuda_fail(e, "cudaEventCreate");
        }
    h->timing = on != 0;
    return ROLLOUT_OK;
}

int dqn_test_stall(dqn_handle *h, int on)
{
    clear_error();
    if (!h) return set_error(ROLLOUT_ERR_INVALID, "null handle");
    h->test_stall = on != 0;
    return ROLLOUT_OK;
}

int dqn_phase_ms(dqn_handle *h, float *ms)
{
    clear_error();
    if (!h || !ms) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (!h->timed_run) return set_error(ROLLOUT_ERR_INVALID, "no timed run");
    cudaError_t e = cudaEventSynchronize(h->ev[3]);
    for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaEventElapsedTime(ms + i, h->ev[i], h->ev[i + 1]);
    return e == cudaSuccess ? ROLLOUT_OK : cuda_fail(e, "cudaEventElapsedTime");
}

int dqn_status(dqn_handle *h)
{
    clear_error();
    if (!h) return set_error(ROLLOUT_ERR_INVALID, "null handle");
    cudaError_t e = cudaStreamSynchronize(h->last_stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int st = 0;
    if ((e = cudaMemcpy(&st, h->d_status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemset(h->d_status, 0, sizeof(int))) != cudaSuccess)
        return cuda_fail(e, "status read");
    return st;
}

void dqn_destroy(dqn_handle *h)
{
    if (!h) return;
    cudaDeviceSynchronize();
    free_handle(h);
}

}  // extern "C"
