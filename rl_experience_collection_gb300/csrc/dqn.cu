// dqn.cu -- the DQN experience collector (include/dqn.h) on tcgen05 tensor
// cores, bf16 operands, float32 accumulation in TMEM.
//
// Page "GPU Pipeline Phase 2b: Zero-Roundtrip CUDA Experience Collection",
// "Data Flow" (steps 1-15) and "Kernel Components" 1 (dueling Q network), 7
// (TD error), 8 (LCG); the environment is the PPO collector's (env.cuh).
//
// A padded copy of the features (rows of kFPad floats, the bar's simple
// return in column 51) is refilled first; then three stream-ordered phases,
// as in the PPO collector:
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
// array V' after the trade.  Episode recycling (dqn_set_recycle) runs second
// builds of the rollout and the target pass: after a done the rollout moves the
// episode to a bar drawn from its LCG and stores every step's bar, which the
// state rows and the target pass read instead of start + t.
//
// Both kernels have 16 row warps (warp w serves TMEM lanes and rows
// 32 (w % 4) .. + 31 and the column quarter w / 4 of every 64-column chunk),
// three producer warps streaming the weights (one per ring stage), one MMA
// warp, and overlap each layer's epilogue with the next layer's MMAs through
// two alternating TMEM regions and per-K-chunk handoffs (see each kernel's
// comment).  Every wait is bounded; a wait that gives up sets a flag that
// ends every role's loop, and the status word records the timeout.
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
constexpr int kStages = 3;
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
    const float *Fpad;   // F with rows padded to kFPad floats; column 51 holds the bar's simple return
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
    int32_t *bars;       // recycling build: the bar of every step (read by the state rows and the target pass)
};

struct TargetArgs {
    const float *F;
    const float *Fpad;   // F with rows padded to kFPad floats (16-byte aligned)
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
    const int32_t *bars; // the bar of every step (episode recycling), or null: start + t
};

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

// ---------------------------------------------------------------------------
// target pass: curiosity and the target network over every transition
//
// Persistent CTAs over tiles of 128 transitions.  Warp roles: 16 row warps
// (warp w serves TMEM lanes / rows 32 (w % 4) .. + 31 and the column quarter
// w / 4 of every 64-column chunk), three producer warps (warp kTProd0 + s fills
// ring stage s), one MMA warp (TMEM allocation; one lane issues), and four
// builder warps that write the next tile's operand rows X and X' while the
// row warps drain the current one.
//
// TMEM holds two 256-column regions.  The j-th tile of a CTA puts target
// layers 1 and 3 and the head into region s = j & 1 and layer 2 into the
// other one, so every layer starts on its first K-chunk while the rows still
// drain the rest of the previous layer, and the next tile's layer 1 runs
// while this tile's layer 3 drains.  The curiosity model takes the 64 columns that a drained
// chunk leaves free: layer 1 at [0, 64) of region s once H1's chunk 0 is out,
// layer 2 at [0, 64) of the other region once H2's chunk 0 is out.  The head
// (N = 48) accumulates into [0, 48) of region s, which H3's chunk 0 frees.
//
// Per tile the MMA lane takes its weight units in this order (the producers
// stream them in the same order): W2 chunk 0, C1, W2 chunks 1-3, W3 chunk 0,
// C2, W3 chunks 1-3, the head, the next tile's W1 (none after the last tile);
// the CTA's first tile is preceded by its W1.
constexpr int kTRowWarps = 16;
constexpr int kTBuilders = 4;                     // X / X' builder warps, 32 rows each
constexpr int kTProd0 = kTRowWarps, kTMma = kTProd0 + kStages, kTBuild0 = kTMma + 1;
constexpr int kTThreads = (kTBuild0 + kTBuilders) * 32;
constexpr int kTUnitsPerTile = 12;

struct TBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t x;             // builders -> MMA: X and X' of a tile are written
    uint64_t h1[4], h2[4], h3[4];   // rows -> MMA: K-chunk c of a hidden layer is in Hb
    uint64_t z;             // rows -> MMA: the curiosity hidden layer Z is written
    uint64_t cz;            // rows -> MMA: curiosity layer 2's columns are read
    uint64_t hd_free;       // quarter-0 row warps -> MMA: the head's columns are read
    uint64_t q1, c1, q2, c2, q3, hd;   // MMA -> rows: that group of MMAs is complete
    uint64_t mse[4];        // quarters 1-3 -> quarter 0 of the same lanes: partial sums written
    uint64_t fin;
};

constexpr int kOneHotLd = 72;                        // bf16 per one-hot row (64 + 8: rows start on different banks)
constexpr int kTFloats = kBiasFloats + 128 + 3 * 128 + 2 * 128 + 2 * 128 + 128;
constexpr int kTSmem = 1024 + 3 * kChunk + 4 * kChunk + kStages * kStage + kTFloats * 4 + kActions * kOneHotLd * 2 + 1024;
static_assert(kTSmem <= 232448, "target pass shared memory");
static_assert(sizeof(TBars) <= 1024, "target pass barriers");

// unit g of a CTA (12 a tile, the last tile's 11 ending with its head): its
// byte offset and size in the weight image (see the order above)
__device__ __forceinline__ void target_unit(const DqnImage &w, long long g, long long &off, uint32_t &bytes)
{
    int u;            // 0 W1, 1-4 W2, 5-8 W3, 9 head, 10 C1, 11 C2
    if (g == 0) {
        u = 0;
    } else {
        const long long k = g - 1, j = k / kTUnitsPerTile;
        int pos = (int)(k - j * kTUnitsPerTile);
        // positions 0..11 -> units 1, 10, 2, 3, 4, 5, 11, 6, 7, 8, 9, 0 (a nibble each)
        u = (int)((0x0987'6B54'32A1ull >> (4 * pos)) & 15u);
    }
    if (u >= 10) {
        off = w.unit_off[kNetUnits] + (u - 10) * kCurTile;
        bytes = kCurTile;
    } else {
        off = w.unit_off[kNetUnits + 1 + u];
        bytes = w.unit_bytes[kNetUnits + 1 + u];
    }
}

// one transition's inputs to the target pass, loaded a tile ahead: every
// address depends on the row index only, so the loads are issued together
struct TMeta {
    long long i;     // flat transition index
    int valid;       // i < N L and the episode's start is in range
    int act, done, start, t, aprev, dprev;
    int bar;         // the bar of the step (0 when !valid)
    float r0, qs, vin, vp;
};

template <bool kRecycle>
__device__ __forceinline__ void load_meta(const TargetArgs &a, long long tile, int r, TMeta &m)
{
    const long long R = (long long)a.N * a.L;
    m.i = tile * 128 + r;
    const long long ic = m.i < R ? m.i : R - 1;
    const long long n = ic <= 0x7fffffffLL ? (long long)((uint32_t)ic / (uint32_t)a.L) : ic / a.L;
    m.t = (int)(ic - n * a.L);
    const long long ip = m.t > 0 ? ic - 1 : ic;
    m.start = __ldg(a.starts + n);
    m.act = a.actions[ic];
    m.done = a.dones[ic];
    m.r0 = a.rewards[ic];
    m.qs = a.q[ic];
    m.vin = a.td[ic];
    m.vp = a.v_post[ic];
    m.aprev = a.actions[ip];
    m.dprev = a.dones[ip];
    if (kRecycle) m.bar = a.bars[ic];
}

// validity and the derived fields, once the loads have landed
template <bool kRecycle>
__device__ __forceinline__ void resolve_meta(const TargetArgs &a, TMeta &m)
{
    const long long R = (long long)a.N * a.L;
    m.valid = m.i < R && start_ok(m.start, a.L, a.n_bars);
    // the one-hot row read stays in bounds whatever the rollout left here
    // (its rows after a give-up are unwritten)
    if (!m.valid || (unsigned)m.act >= (unsigned)kActions) m.act = 0;
    // a stored bar (episode recycling) is read where the rollout wrote it; the
    // feature reads stay in bounds whatever a rollout that gave up left behind
    if (!kRecycle) m.bar = m.start + m.t;
    if (!m.valid || (unsigned)m.bar > (unsigned)(a.n_bars - 2)) m.bar = 0;
}

// the market columns of [16 q, 16 q + 16) of a padded feature row (zero past
// column 50 or when !valid), in 16-byte loads; state16_tail then fills V, e,
// spread into columns 51-53
__device__ __forceinline__ void feat16(const float *Fprow, int q, bool valid, float (&v)[16])
{
    const float4 *src = reinterpret_cast<const float4 *>(Fprow) + 4 * q;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float4 f = make_float4(0.f, 0.f, 0.f, 0.f);
        if (valid && 16 * q + 4 * k < kMarket) f = __ldg(src + k);
        v[4 * k + 0] = f.x;
        v[4 * k + 1] = f.y;
        v[4 * k + 2] = f.z;
        v[4 * k + 3] = f.w;
    }
    if (q == 3) v[kMarket - 48] = 0.f;   // column 51 of the padded row is not a market column
}

__device__ __forceinline__ void state16_tail(float V, float e, float spread, int q, bool valid, float (&v)[16])
{
    if (q == 3 && valid) {
        v[kMarket - 48] = V;
        v[kMarket + 1 - 48] = e;
        v[kMarket + 2 - 48] = spread;
    }
}

// one whole operand row: [F[b, 0..50], V, e, spread, 0 x 10] rounded to bf16
// into row r of a 64-column 128-byte-swizzled tile (zeros when !valid); Fprow
// is the padded feature row (13 16-byte loads, in flight together)
__device__ __forceinline__ void state_row(uint8_t *tile, int r, const float *Fprow, bool valid, float V, float e,
                                          float spread)
{
    const float4 *src = reinterpret_cast<const float4 *>(Fprow);
    float4 f[13];
#pragma unroll
    for (int k = 0; k < 13; ++k) f[k] = valid ? __ldg(src + k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int u = 0; u < 6; ++u) {
        uint4 p;
        p.x = pack_bf16x2(f[2 * u].x, f[2 * u].y);
        p.y = pack_bf16x2(f[2 * u].z, f[2 * u].w);
        p.z = pack_bf16x2(f[2 * u + 1].x, f[2 * u + 1].y);
        p.w = pack_bf16x2(f[2 * u + 1].z, f[2 * u + 1].w);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(r, u)) = p;
    }
    uint4 p;
    p.x = pack_bf16x2(f[12].x, f[12].y);
    p.y = pack_bf16x2(f[12].z, valid ? V : 0.f);
    p.z = valid ? pack_bf16x2(e, spread) : 0u;
    p.w = 0u;
    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 6)) = p;
    *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 7)) = make_uint4(0u, 0u, 0u, 0u);
}

// 16 values rounded to bf16 into a 128-byte-swizzled operand chunk, at the
// byte offsets of the row's two 16-byte units (sw128_offset)
__device__ __forceinline__ void put16(uint8_t *chunk, uint32_t off0, uint32_t off1, const float (&v)[16])
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 p;
        p.x = pack_bf16x2(v[8 * h + 0], v[8 * h + 1]);
        p.y = pack_bf16x2(v[8 * h + 2], v[8 * h + 3]);
        p.z = pack_bf16x2(v[8 * h + 4], v[8 * h + 5]);
        p.w = pack_bf16x2(v[8 * h + 6], v[8 * h + 7]);
        *reinterpret_cast<uint4 *>(chunk + (h ? off1 : off0)) = p;
    }
}

__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16])
{
    uint32_t x[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
          "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15])
        : "r"(taddr)
        : "memory");
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(x[i]);
}

// 16 accumulator columns + bias (16-byte aligned), LeakyReLU, bf16 into the
// operand chunk; max(y, 0.01 y) is LeakyReLU(0.01) exactly, signed zeros included
__device__ __forceinline__ void drain16_leaky(uint32_t taddr, const float *bias, uint8_t *chunk, uint32_t off0,
                                              uint32_t off1)
{
    float v[16];
    tmem_ld16(taddr, v);
    const float4 *b4 = reinterpret_cast<const float4 *>(bias);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const float4 b = b4[k];
        v[4 * k + 0] += b.x;
        v[4 * k + 1] += b.y;
        v[4 * k + 2] += b.z;
        v[4 * k + 3] += b.w;
    }
#pragma unroll
    for (int k = 0; k < 16; ++k) v[k] = fmaxf(v[k], 0.01f * v[k]);
    put16(chunk, off0, off1, v);
}

// one arrival per warp after every lane's shared-memory writes and TMEM reads
__device__ __forceinline__ void publish(uint64_t *bar)
{
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// kStall: a test build in which the first producer of CTA 0 issues no copy, so
// that CTA's MMA issuer waits on a weight stage that never fills and the
// bounded-wait exit runs (dqn_test_stall).  kRecycle: every step's bar is the
// one the rollout stored (episode recycling), and a done step's next state is
// never the next row's.
template <bool kStall, bool kRecycle>
__global__ void __launch_bounds__(kTThreads, 1) dqn_target_kernel(TargetArgs a, DqnImage w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *X = base, *Xn = X + kChunk, *Z = Xn + kChunk;
    uint8_t *Hb = Z + kChunk;
    uint8_t *ring = Hb + 4 * kChunk;
    float *bias = reinterpret_cast<float *>(ring + kStages * kStage);
    float *cb1 = bias + kBiasFloats, *cb2 = cb1 + 64;
    float *mse_part = cb2 + 64;                        // [3][128]: curiosity partial sums of quarters 1-3
    float *hsum = mse_part + 3 * 128;                  // [2][128]: advantage partial sums of quarters 1, 2
    float *hmax = hsum + 2 * 128;                      // [2][128]: advantage partial maxima of quarters 1, 2
    float *hval = hmax + 2 * 128;                      // [128]: V (quarter 2)
    uint16_t *onehot = reinterpret_cast<uint16_t *>(hval + 128);   // [45][kOneHotLd] bf16 C1[:, 54 + a]
    TBars *bars = reinterpret_cast<TBars *>(onehot + kActions * kOneHotLd);
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->x, kTBuilders);
        for (int c = 0; c < 4; ++c) {
            mbar_init(&bars->h1[c], kTRowWarps);
            mbar_init(&bars->h2[c], kTRowWarps);
            mbar_init(&bars->h3[c], kTRowWarps);
            mbar_init(&bars->mse[c], 3);
        }
        mbar_init(&bars->z, kTRowWarps);
        mbar_init(&bars->cz, kTRowWarps);
        mbar_init(&bars->hd_free, 12);
        mbar_init(&bars->q1, 1);
        mbar_init(&bars->c1, 1);
        mbar_init(&bars->q2, 1);
        mbar_init(&bars->c2, 1);
        mbar_init(&bars->q3, 1);
        mbar_init(&bars->hd, 1);
        mbar_init(&bars->fin, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < kBiasFloats; i += kTThreads) bias[i] = w.target_bias[i];
    for (int i = tid; i < 64; i += kTThreads) {
        cb1[i] = w.cur_b1[i];
        cb2[i] = w.cur_b2[i];
    }
    // the one-hot columns are bf16 values already: their upper halves are exact
    for (int i = tid; i < kActions * 64; i += kTThreads)
        onehot[(i >> 6) * kOneHotLd + (i & 63)] = (uint16_t)(__float_as_uint(w.cur_onehot[i]) >> 16);
    if (warp == kTMma) {
        tmem_alloc(&tmem_base_s, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const long long R = (long long)a.N * a.L;
    const long long n_tiles = (R + 127) / 128;

    if (warp < kTRowWarps) {
        // ------------------------------------------------------------ rows
        const int quad = warp & 3, q = warp >> 2, r = quad * 32 + lane;
        const uint32_t lane_t = tmem + ((uint32_t)(quad * 32) << 16) + 16 * q;
        const uint32_t off0 = sw128_offset(r, 2 * q), off1 = sw128_offset(r, 2 * q + 1);
        uint32_t it = 0;
        bool ok = true;
        auto wait = [&](uint64_t *bar) {
            ok = ok && warp_wait(bar, it & 1, &abort_flag);
            tc_fence_after();
        };
        TMeta cur;
        for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
            const uint32_t rs = (it & 1) * 256, ro = 256 - rs;
            load_meta<kRecycle>(a, tile, r, cur);                    // first used by curiosity layer 1
            // layer 1 of the target net (region s) -> H1, chunk by chunk
            wait(&bars->q1);
            if (!ok) break;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                drain16_leaky(lane_t + rs + 64 * c, bias + 64 * c + 16 * q, Hb + c * kChunk, off0, off1);
                publish(&bars->h1[c]);
            }
            // x' (this quarter's columns, float32) for the curiosity error, in
            // flight until curiosity layer 2; issued before the builders' loads
            // of the next tile begin (they wait for curiosity layer 1)
            resolve_meta<kRecycle>(a, cur);
            float xn[16];
            {
                const long long b = cur.bar;
                feat16(a.Fpad + (b + 1) * kFPad, q, cur.valid, xn);
                state16_tail(cur.vp, exposure_of(cur.act), a.env.spread, q, cur.valid, xn);
            }
            // curiosity layer 1 ([0, 64) of region s): Z = ReLU(X C1^T + c1 + C1[:, 54 + a])
            wait(&bars->c1);
            if (!ok) break;
            {
                float v[16];
                tmem_ld16(lane_t + rs, v);
                const uint4 *oh = reinterpret_cast<const uint4 *>(onehot + cur.act * kOneHotLd + 16 * q);
                const float4 *b4 = reinterpret_cast<const float4 *>(cb1 + 16 * q);
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const uint4 o = oh[h];
                    const uint32_t ow[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const float2 of = unpack_bf16x2(ow[k]);
                        const int j = 8 * h + 2 * k;
                        const float4 b = b4[j >> 2];
                        const float b0 = (j & 3) ? b.z : b.x, b1 = (j & 3) ? b.w : b.y;
                        v[j] = relu(v[j] + b0 + of.x);
                        v[j + 1] = relu(v[j + 1] + b1 + of.y);
                    }
                }
                put16(Z, off0, off1, v);
            }
            publish(&bars->z);
            // layer 2 (the other region) -> H2
            wait(&bars->q2);
            if (!ok) break;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                drain16_leaky(lane_t + ro + 64 * c, bias + kH + 64 * c + 16 * q, Hb + c * kChunk, off0, off1);
                publish(&bars->h2[c]);
            }
            // curiosity layer 2 ([0, 64) of the other region): squared error
            // against x' over the 54 state columns
            wait(&bars->c2);
            if (!ok) break;
            float part = 0.f;
            {
                float v[16];
                tmem_ld16(lane_t + ro, v);
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (16 * q + k < kState) {
                        const float dlt = (v[k] + cb2[16 * q + k]) - xn[k];
                        part += dlt * dlt;
                    }
            }
            publish(&bars->cz);
            if (q != 0) mse_part[(q - 1) * 128 + r] = part;
            if (q == 3) {                                   // no head columns: its share is complete
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->mse[quad]);
            }
            if (a.next_states && cur.i < R) {
                float *dst = a.next_states + cur.i * kState + 16 * q;
#pragma unroll
                for (int k = 0; k < 16; ++k)
                    if (16 * q + k < kState) dst[k] = cur.valid ? xn[k] : 0.f;
            }
            // layer 3 (region s) -> H3
            wait(&bars->q3);
            if (!ok) break;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {
                drain16_leaky(lane_t + rs + 64 * c, bias + 2 * kH + 64 * c + 16 * q, Hb + c * kChunk, off0,
                              off1);
                publish(&bars->h3[c]);
            }
            // the head ([0, 48) of region s); every warp waits for it, since the
            // next tile's H1 overwrites the H3 it reads
            wait(&bars->hd);
            if (!ok) break;
            if (q < 3) {
                // advantage columns 16 q .. 16 q + 15 (V at column 45): this
                // quarter's sum (in column order) and maximum of A_j = D_j + b_j.
                // Q_j = V + (A_j - mean A) is nondecreasing in A_j under float
                // rounding, so max_j Q_j = V + (max_j A_j - mean A) exactly.
                // The TMEM load is warp-wide (.sync.aligned): every lane issues it,
                // rows past the end included; only stores are per row.
                float d[16], sA = 0.f, mA = -INFINITY, V = 0.f;
                tmem_ld16(lane_t + rs, d);
                publish(&bars->hd_free);
                const float *bh = bias + 3 * kH + 16 * q;
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    const int j = 16 * q + k;
                    const float A = d[k] + bh[k];
                    if (j < kActions) {
                        sA += A;
                        mA = fmaxf(mA, A);
                    } else if (j == kActions) {
                        V = A;
                    }
                }
                if (q > 0) {
                    hsum[(q - 1) * 128 + r] = sA;
                    hmax[(q - 1) * 128 + r] = mA;
                    if (q == 2) hval[r] = V;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&bars->mse[quad]);
                } else {
                    ok = warp_wait(&bars->mse[quad], it & 1, &abort_flag);
                    if (!ok) break;
                    const float sumA = (sA + hsum[r]) + hsum[128 + r];
                    const float maxA = fmaxf(fmaxf(mA, hmax[r]), hmax[128 + r]);
                    const float Vh = hval[r];
                    const float meanA = sumA / (float)kActions;
                    const float qmax = Vh + (maxA - meanA);
                    const float mse = part + mse_part[r] + mse_part[128 + r] + mse_part[256 + r];
                    const float cur_bonus = a.env.cur_coef * (mse / (float)kState);
                    if (cur.valid) {
                        const float rew = cur.r0 + cur_bonus;
                        a.rewards[cur.i] = rew;
                        a.td[cur.i] = fabsf(rew + a.gamma * qmax * (1.f - (float)cur.done) - cur.qs);
                    } else if (cur.i < R) {
                        a.rewards[cur.i] = 0.f;
                        a.td[cur.i] = 0.f;
                    }
                }
            }
        }
    } else if (warp < kTMma) {
        // ------------------------------------------------------------ weight stream, stage st
        const int st = warp - kTProd0;
        if (lane == 0) {
            const long long n_my = n_tiles > blockIdx.x ? (n_tiles - 1 - blockIdx.x) / gridDim.x + 1 : 0;
            const long long total = (kStall && blockIdx.x == 0 && st == 0) ? 0 : kTUnitsPerTile * n_my;
            long long last = -1;
            for (long long u = st; u < total; u += kStages) {
                long long off;
                uint32_t bytes;
                target_unit(w, u, off, bytes);
                if (u >= kStages && !mbar_wait(&bars->empty[st], (uint32_t)((u / kStages - 1) & 1), &abort_flag))
                    break;
                mbar_arrive_expect_tx(&bars->full[st], bytes);
                bulk_g2s(ring + st * kStage, w.base + off, bytes, &bars->full[st]);
                last = u;
            }
            // its last copy completes before the CTA may exit
            if (last >= 0) mbar_wait_drain(&bars->full[st], (uint32_t)((last / kStages) & 1));
        }
    } else if (warp >= kTBuild0) {
        // ------------------------------------------------------------ X and X' builders
        // Build a tile's operand rows while the row warps drain the previous
        // tile, builder w taking rows 32 w .. 32 w + 31: X = the state rows; X'
        // = the pre-reset next states, whose market columns are those of the
        // next row of X (the same rounding of the same bar) wherever that row is
        // the same episode's next step and this warp's own, and otherwise come
        // from the feature matrix.  X and X' of the previous tile are free once
        // its layer 1 and curiosity layer 1 are complete.
        const int r = 32 * (warp - kTBuild0) + lane;
        uint32_t it = 0;
        bool ok = true;
        for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
            if (it > 0) {
                ok = warp_wait(&bars->q1, (it - 1) & 1, &abort_flag);
                ok = ok && warp_wait(&bars->c1, (it - 1) & 1, &abort_flag);
                if (!ok) break;
            }
            TMeta m;
            load_meta<kRecycle>(a, tile, r, m);
            resolve_meta<kRecycle>(a, m);
            const long long b = m.bar;
            const float e_in = (m.t == 0 || m.dprev) ? 0.f : exposure_of(m.aprev);
            // the warp's 32 rows are consecutive bars of one episode: their
            // padded feature rows are one contiguous run, read in whole lines
            const long long b0 = __shfl_sync(0xffffffffu, b, 0);
            if (__all_sync(0xffffffffu, m.valid && b == b0 + lane)) {
                const float4 *run = reinterpret_cast<const float4 *>(a.Fpad + b0 * kFPad);
#pragma unroll
                for (int h = 0; h < 2; ++h) {                  // two batches of loads in flight (registers)
                    const int j0 = h ? 7 : 0, j1 = h ? 13 : 7;
                    float4 f[7];
#pragma unroll
                    for (int j = 0; j < 7; ++j)
                        if (j0 + j < j1) f[j] = __ldg(run + 32 * (j0 + j) + lane);
#pragma unroll
                    for (int jj = 0; jj < 7; ++jj) {
                        const int j = j0 + jj;
                        if (j >= j1) break;
                        const float4 v = f[jj];
                        const int idx = 32 * j + lane, rr = idx / 13, c4 = idx - 13 * rr;   // columns 4 c4 .. + 3
                        const float Vr = __shfl_sync(0xffffffffu, m.vin, rr);
                        uint2 p;
                        p.x = pack_bf16x2(v.x, v.y);
                        p.y = pack_bf16x2(v.z, c4 == 12 ? Vr : v.w);                   // column 51 is V
                        *reinterpret_cast<uint2 *>(X + sw128_offset(32 * (warp - kTBuild0) + rr, c4 >> 1) +
                                                   8 * (c4 & 1)) = p;
                    }
                }
                // columns 52..63 of the lane's own row: e, spread, zeros
                *reinterpret_cast<uint2 *>(X + sw128_offset(r, 6) + 8) = make_uint2(pack_bf16x2(e_in, a.env.spread), 0u);
                *reinterpret_cast<uint4 *>(X + sw128_offset(r, 7)) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                state_row(X, r, a.Fpad + b * kFPad, m.valid, m.vin, e_in, a.env.spread);
            }
            __syncwarp();                                  // the warp's rows of X are written
            // (with recycling a done step's next row starts a new episode elsewhere)
            if (m.valid && lane < 31 && m.t < a.L - 1 && !(kRecycle && m.done)) {
#pragma unroll
                for (int u = 0; u < 6; ++u)
                    *reinterpret_cast<uint4 *>(Xn + sw128_offset(r, u)) =
                        *reinterpret_cast<const uint4 *>(X + sw128_offset(r + 1, u));
                const uint4 w6 = *reinterpret_cast<const uint4 *>(X + sw128_offset(r + 1, 6));
                uint4 p;
                p.x = w6.x;                                                           // columns 48, 49
                p.y = (w6.y & 0xFFFFu) | (pack_bf16x2(0.f, m.vp) & 0xFFFF0000u);       // 50, V'
                p.z = pack_bf16x2(exposure_of(m.act), a.env.spread);                  // e', spread
                p.w = 0u;
                *reinterpret_cast<uint4 *>(Xn + sw128_offset(r, 6)) = p;
                *reinterpret_cast<uint4 *>(Xn + sw128_offset(r, 7)) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                state_row(Xn, r, a.Fpad + (b + 1) * kFPad, m.valid, m.vp, exposure_of(m.act), a.env.spread);
            }
            publish(&bars->x);
        }
    } else {
        // ------------------------------------------------------------ MMA issue
        if (lane == 0) {
            const uint32_t id256 = idesc(true, 128, kH), id48 = idesc(true, 128, kHeadN), id64 = idesc(true, 128, 64);
            const uint32_t sX = smem_u32(X), sXn = smem_u32(Xn), sZ = smem_u32(Z), sH = smem_u32(Hb);
            const uint32_t sRing = smem_u32(ring);
            long long g = 0;      // weight units taken
            uint32_t it = 0;
            bool ok = true;
            auto take = [&]() -> uint32_t {
                const int st = (int)(g % kStages);
                ok = ok && mbar_wait(&bars->full[st], (uint32_t)((g / kStages) & 1), &abort_flag);
                tc_fence_after();
                return sRing + st * kStage;
            };
            auto release = [&]() {
                mma_commit(&bars->empty[g % kStages]);
                ++g;
            };
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                ok = ok && mbar_wait(bar, parity, &abort_flag);
                tc_fence_after();
            };
            // D[col] (+)= A(one 64-column K-chunk at a) B(b)^T
            auto chunk = [&](uint32_t col, uint32_t a_s, uint32_t b_s, uint32_t id, bool accumulate) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma<true>(tmem + col, desc_sw128(a_s + 32 * k), desc_sw128(b_s + 32 * k), id,
                              (accumulate || k > 0) ? 1u : 0u);
            };
            for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x, ++it) {
                const uint32_t rs = (it & 1) * 256, ro = 256 - rs, par = it & 1;
                const bool has_next = tile + gridDim.x < n_tiles;
                uint32_t u;
                if (it == 0) {
                    u = take();
                    wait(&bars->x, 0);
                    if (!ok) break;
                    chunk(rs, sXn, u, id256, false);
                    release();
                    mma_commit(&bars->q1);
                }
                // layer 2 into the other region; the previous tile's head was there
                u = take();
                wait(&bars->h1[0], par);
                if (it > 0) wait(&bars->hd_free, par ^ 1u);
                if (!ok) break;
                chunk(ro, sH, u, id256, false);
                release();
                // curiosity layer 1 into [0, 64) of region s, which H1's chunk 0 has left
                u = take();
                if (!ok) break;
                chunk(rs, sX, u, id64, false);
                release();
                mma_commit(&bars->c1);
                for (int c = 1; c < 4 && ok; ++c) {
                    u = take();
                    wait(&bars->h1[c], par);
                    if (!ok) break;
                    chunk(ro, sH + c * kChunk, u, id256, true);
                    release();
                }
                if (!ok) break;
                mma_commit(&bars->q2);
                // layer 3 into region s (H1 and curiosity layer 1 are out of it)
                u = take();
                wait(&bars->h2[0], par);
                if (!ok) break;
                chunk(rs, sH, u, id256, false);
                release();
                // curiosity layer 2 into [0, 64) of the other region, which H2's chunk 0 has left
                u = take();
                wait(&bars->z, par);
                if (!ok) break;
                chunk(ro, sZ, u, id64, false);
                release();
                mma_commit(&bars->c2);
                for (int c = 1; c < 4 && ok; ++c) {
                    u = take();
                    wait(&bars->h2[c], par);
                    if (!ok) break;
                    chunk(rs, sH + c * kChunk, u, id256, true);
                    release();
                }
                if (!ok) break;
                mma_commit(&bars->q3);
                // the head into [0, 48) of region s, K-chunk by K-chunk as H3 comes out
                u = take();
                for (int c = 0; c < 4 && ok; ++c) {
                    wait(&bars->h3[c], par);
                    if (!ok) break;
                    chunk(rs, sH + c * kChunk, u + c * kHeadTile, id48, c > 0);
                }
                if (!ok) break;
                release();
                mma_commit(&bars->hd);
                // the next tile's layer 1 into the other region, once H2 and
                // curiosity layer 2 are out of it and the builders have written X'
                if (has_next) {
                    u = take();
                    wait(&bars->cz, par);
                    wait(&bars->x, par ^ 1u);
                    if (!ok) break;
                    chunk(ro, sXn, u, id256, false);
                    release();
                    mma_commit(&bars->q1);
                }
            }
            // every MMA issued has completed before TMEM is freed
            mma_commit(&bars->fin);
            mbar_wait_drain(&bars->fin, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTMma) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
    if (tid == 0 && abort_flag) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
}

// two K-chunks (16 accumulator columns each, at taddr0 and taddr1) loaded
// together, then each + bias, LeakyReLU, bf16 into its operand chunk and
// published on its barrier: one TMEM round trip for two chunks
__device__ __forceinline__ void drain_pair_leaky(uint32_t taddr0, uint32_t taddr1, const float *bias0,
                                                 const float *bias1, uint8_t *chunk0, uint8_t *chunk1, uint32_t off0,
                                                 uint32_t off1, uint64_t *bar0, uint64_t *bar1)
{
    uint32_t x[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(x[0]), "=r"(x[1]), "=r"(x[2]), "=r"(x[3]), "=r"(x[4]), "=r"(x[5]), "=r"(x[6]), "=r"(x[7]),
          "=r"(x[8]), "=r"(x[9]), "=r"(x[10]), "=r"(x[11]), "=r"(x[12]), "=r"(x[13]), "=r"(x[14]), "=r"(x[15])
        : "r"(taddr0)
        : "memory");
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(x[16]), "=r"(x[17]), "=r"(x[18]), "=r"(x[19]), "=r"(x[20]), "=r"(x[21]), "=r"(x[22]), "=r"(x[23]),
          "=r"(x[24]), "=r"(x[25]), "=r"(x[26]), "=r"(x[27]), "=r"(x[28]), "=r"(x[29]), "=r"(x[30]), "=r"(x[31])
        : "r"(taddr1)
        : "memory");
    tmem_ld_wait();
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const float4 *b4 = reinterpret_cast<const float4 *>(h ? bias1 : bias0);
        float v[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 b = b4[k];
            v[4 * k + 0] = __uint_as_float(x[16 * h + 4 * k + 0]) + b.x;
            v[4 * k + 1] = __uint_as_float(x[16 * h + 4 * k + 1]) + b.y;
            v[4 * k + 2] = __uint_as_float(x[16 * h + 4 * k + 2]) + b.z;
            v[4 * k + 3] = __uint_as_float(x[16 * h + 4 * k + 3]) + b.w;
        }
#pragma unroll
        for (int k = 0; k < 16; ++k) v[k] = fmaxf(v[k], 0.01f * v[k]);
        put16(h ? chunk1 : chunk0, off0, off1, v);
        publish(h ? bar1 : bar0);
    }
}

// ---------------------------------------------------------------------------
// rollout: the online network inside the serial step loop
//
// A CTA steps 128 episodes (one per TMEM lane / operand row) through all L
// bars.  Warp roles: 16 row warps (warp w serves TMEM lanes / rows
// 32 (w % 4) .. + 31 and the column quarter w / 4 of every 64-column chunk),
// three producer warps (warp kRProd0 + s fills ring stage s), one MMA warp.
// TMEM holds two 256-column regions; step t puts layers 1 and 3 and the head
// into region s = t & 1 and layer 2 into the other one, so each layer starts
// on its first K-chunk while the rows still drain the rest of the previous
// one.  The head accumulates into [0, 48) of region s (freed by H3's chunk 0).
// The market columns of the next step's state rows are known a step ahead
// (the bar advances by one whatever the action): warps of quarters 1-3 write
// columns 0-47 of X as soon as layer 1 has read it.  The head's 48 columns
// are read by the quarter 0-2 warps, 16 each: each forms its advantage sum and
// first maximum, quarters 1 and 2 pass theirs through shared memory, and the
// quarter-0 warps, which hold the episodes' environment state, combine them,
// pick the action, step the environment and write columns 48-55 (F[.., 48..50],
// V, e, spread).  The next step's layer 1 is issued in two parts: its three
// K16 steps over the market columns before this step's head, its last one
// (columns 48-63) once the quarter-0 warps have written them.  Per step the
// MMA lane takes its weight units in this order (the producers stream them in
// the same order): W2 chunks 0-3, W3 chunks 0-3, the next step's W1 (streamed
// but unused after the last step), the head; the first step is preceded by
// its W1.
constexpr int kRRowWarps = 16;
constexpr int kRProd0 = kRRowWarps, kRMma = kRProd0 + kStages, kRThreads = (kRMma + 1) * 32;
constexpr int kRUnitsPerStep = 10;

struct RBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t xm, xt;        // rows -> MMA: X of a step is written, market columns 0..47 (the
                            // quarter 1-3 warps) and columns 48..63 (the quarter-0 warps)
    uint64_t h1[4], h2[4], h3[4];   // rows -> MMA: K-chunk c of a hidden layer is in Hb
    uint64_t hd_free;       // quarter 0-2 row warps -> MMA: the head's columns are read
    uint64_t q1, q2, q3, hd;        // MMA -> rows: that layer's MMAs are complete
    uint64_t hx2[4];                // quarters 1, 2 -> quarter 0 of the same lanes: head partials written
    uint64_t ve;                    // recycling build: quarter 0 -> the others: the next step's bar and LCG state
    uint64_t fin;
};

// head exchange: sums [2][128], V [128], best [2][128], max [2][128], A(a_rand) [128];
// recycling: the next step's bar [128] and LCG state [128]
constexpr int kRXFloats = 10 * 128;
constexpr int kRSmem =
    1024 + kChunk + 4 * kChunk + kStages * kStage + kBiasFloats * 4 + kDivWords * 4 + kRXFloats * 4 + 1024;
static_assert(kRSmem <= 232448, "rollout shared memory");
static_assert(sizeof(RBars) <= 1024, "rollout barriers");

// unit g of the rollout's weight stream (10 a step, and one more W1 after the
// last step's W3, unused): its index in the image
__device__ __forceinline__ int rollout_unit(long long g)
{
    if (g == 0) return 0;                                  // the first step's W1
    const int pos = (int)((g - 1) % kRUnitsPerStep);       // W2 0-3, W3 0-3, next W1, head
    return pos < 8 ? 1 + pos : (pos == 8 ? 0 : 9);
}

// kRecycle: episode recycling (after a done, the next step starts at a fresh bar
// drawn from the episode's LCG); the quarter-0 warps, which step the
// environment, pass each row's next bar and LCG state to the other warps
template <bool kRecycle>
__global__ void __launch_bounds__(kRThreads, 1) dqn_rollout_kernel(RolloutArgs a, DqnImage w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *X = base;                          // 1 K-chunk
    uint8_t *Hb = X + kChunk;                   // 4 K-chunks
    uint8_t *ring = Hb + 4 * kChunk;
    float *bias = reinterpret_cast<float *>(ring + kStages * kStage);
    uint32_t *div_s = reinterpret_cast<uint32_t *>(bias + kBiasFloats);
    float *hsum = reinterpret_cast<float *>(div_s + kDivWords);      // [2][128] advantage sums of quarters 1, 2
    float *hval = hsum + 2 * 128;                                     // [128] V (quarter 2)
    int *hbest = reinterpret_cast<int *>(hval + 128);                 // [2][128] first maximum's column, quarters 1, 2
    float *hqmax = reinterpret_cast<float *>(hbest + 2 * 128);        // [2][128] their maxima of A
    float *hqrand = hqmax + 2 * 128;                                  // [128] A of the random action (quarters 1, 2)
    int *bar_s = reinterpret_cast<int *>(hqrand + 128);               // [128] recycling: the row's next bar
    uint32_t *rng_s = reinterpret_cast<uint32_t *>(bar_s + 128);      // [128] recycling: the row's LCG state
    RBars *bars = reinterpret_cast<RBars *>(rng_s + 128);
    __shared__ uint32_t tmem_base_s;
    __shared__ volatile int abort_flag;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&bars->full[s], 1);
            mbar_init(&bars->empty[s], 1);
        }
        mbar_init(&bars->xm, kRRowWarps - 4);
        mbar_init(&bars->xt, 4);
        for (int c = 0; c < 4; ++c) {
            mbar_init(&bars->h1[c], kRRowWarps);
            mbar_init(&bars->h2[c], kRRowWarps);
            mbar_init(&bars->h3[c], kRRowWarps);
        }
        mbar_init(&bars->hd_free, 12);
        for (int k = 0; k < 4; ++k) mbar_init(&bars->hx2[k], 2);
        mbar_init(&bars->ve, 4);
        mbar_init(&bars->q1, 1);
        mbar_init(&bars->q2, 1);
        mbar_init(&bars->q3, 1);
        mbar_init(&bars->hd, 1);
        mbar_init(&bars->fin, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    for (int i = tid; i < kBiasFloats; i += kRThreads) bias[i] = w.online_bias[i];
    for (int i = tid; i < kDivWords; i += kRThreads) div_s[i] = a.env.div_low[i];
    if (warp == kRMma) {
        tmem_alloc(&tmem_base_s, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    EnvConst env = a.env;
    env.div_low = div_s;
    const int L = a.L;

    if (warp < kRRowWarps) {
        // ------------------------------------------------------------ rows
        const int quad = warp & 3, q = warp >> 2, r = quad * 32 + lane;
        const int n = blockIdx.x * 128 + r;
        const uint32_t lane_t = tmem + ((uint32_t)(quad * 32) << 16) + 16 * q;
        const uint32_t off0 = sw128_offset(r, 2 * q), off1 = sw128_offset(r, 2 * q + 1);
        // the columns this warp writes into X: quarters 1-3 columns 16 (q - 1) ..
        // + 15 (units 2 (q - 1), 2 (q - 1) + 1); quarter 0 unit 6 (and unit 7, zero)
        const uint32_t xo0 = sw128_offset(r, q > 0 ? 2 * (q - 1) : 6), xo1 = sw128_offset(r, q > 0 ? 2 * q - 1 : 7);
        int start = 0;
        bool valid = n < a.N;
        if (valid) {
            start = a.starts[n];
            if (!start_ok(start, L, a.n_bars)) {
                valid = false;
                if (q == 0) set_status(a.status, ROLLOUT_ERR_RANGE);
            }
        }
        EpState s;
        ep_reset(s);
        s.rng = n < a.N ? a.seeds[n] : 0u;
        long long bar = valid ? start : 0;            // the bar of the current step
        // X columns of bar b: quarters 1-3 their 16 market columns; quarter 0
        // F[b, 48..50] and the bar's simple return (column 51 of the padded row)
        auto fetch = [&](long long b, float (&f)[16]) {
            const float4 *src = reinterpret_cast<const float4 *>(a.Fpad + b * kFPad);
            if (q > 0) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float4 v = valid ? __ldg(src + 4 * (q - 1) + k) : make_float4(0.f, 0.f, 0.f, 0.f);
                    f[4 * k + 0] = v.x;
                    f[4 * k + 1] = v.y;
                    f[4 * k + 2] = v.z;
                    f[4 * k + 3] = v.w;
                }
            } else {
                const float4 v = valid ? __ldg(src + 12) : make_float4(0.f, 0.f, 0.f, 0.f);
                f[0] = v.x;
                f[1] = v.y;
                f[2] = v.z;
                f[3] = v.w;
            }
        };
        // quarter 0's unit 6: F[.., 48..50], V, e, spread, 0, 0 (zero when !valid)
        auto put_tail = [&](const float (&f)[16]) {
            uint4 p;
            p.x = pack_bf16x2(f[0], f[1]);
            p.y = pack_bf16x2(f[2], valid ? s.V : 0.f);
            p.z = valid ? pack_bf16x2(s.e, env.spread) : 0u;
            p.w = 0u;
            *reinterpret_cast<uint4 *>(X + xo0) = p;
        };
        float f[16];
        // X of step 0
        fetch(valid ? start : 0, f);
        if (q > 0) {
            put16(X, xo0, xo1, f);
        } else {
            put_tail(f);
            *reinterpret_cast<uint4 *>(X + xo1) = make_uint4(0u, 0u, 0u, 0u);
        }
        publish(q > 0 ? &bars->xm : &bars->xt);
        bool ok = true;
        for (int t = 0; t < L && ok; ++t) {
            const uint32_t par = t & 1, rs = par * 256, ro = 256 - rs;
            auto wait = [&](uint64_t *bar) {
                ok = ok && warp_wait(bar, par, &abort_flag);
                tc_fence_after();
            };
            // the next bar: X of step t + 1, its return.  With recycling the other
            // quarters learn this step's bar from the quarter-0 warp only after
            // layer 1; they fetch for the bar after the previous one meanwhile and
            // fetch again where the episode was recycled.
            const long long guess = (kRecycle && q > 0 && t > 0) ? bar + 1 : bar;
            if (!kRecycle) bar = valid ? (long long)start + t : 0;
            fetch(valid ? (kRecycle ? guess : bar) + 1 : 0, f);
            // layer 1 (region s) -> H1
            wait(&bars->q1);
            if (!ok) break;
            if (kRecycle && q > 0 && t > 0) {
                // this step's bar and LCG state as the quarter-0 warp left them
                ok = warp_wait(&bars->ve, par ^ 1u, &abort_flag);
                if (!ok) break;
                bar = bar_s[r];
                s.rng = rng_s[r];
                if (bar != guess) fetch(valid ? bar + 1 : 0, f);
            }
#pragma unroll 1
            for (int c = 0; c < 4; c += 2)
                drain_pair_leaky(lane_t + rs + 64 * c, lane_t + rs + 64 * c + 64, bias + 64 * c + 16 * q,
                                 bias + 64 * c + 64 + 16 * q, Hb + c * kChunk, Hb + (c + 1) * kChunk, off0, off1,
                                 &bars->h1[c], &bars->h1[c + 1]);
            // layer 1 has read X: quarters 1-3 write the next step's market columns
            if (q > 0) {
                put16(X, xo0, xo1, f);
                publish(&bars->xm);
            }
            // layer 2 (the other region) -> H2
            wait(&bars->q2);
            if (!ok) break;
#pragma unroll 1
            for (int c = 0; c < 4; c += 2)
                drain_pair_leaky(lane_t + ro + 64 * c, lane_t + ro + 64 * c + 64, bias + kH + 64 * c + 16 * q,
                                 bias + kH + 64 * c + 64 + 16 * q, Hb + c * kChunk, Hb + (c + 1) * kChunk, off0, off1,
                                 &bars->h2[c], &bars->h2[c + 1]);
            // layer 3 (region s) -> H3
            wait(&bars->q3);
            if (!ok) break;
#pragma unroll 1
            for (int c = 0; c < 4; c += 2)
                drain_pair_leaky(lane_t + rs + 64 * c, lane_t + rs + 64 * c + 64, bias + 2 * kH + 64 * c + 16 * q,
                                 bias + 2 * kH + 64 * c + 64 + 16 * q, Hb + c * kChunk, Hb + (c + 1) * kChunk, off0, off1,
                                 &bars->h3[c], &bars->h3[c + 1]);
            if (q == 3) continue;
            // ---- quarters 0-2: the head ([0, 48) of region s): A = columns
            // 0..44, V = column 45; Q_j = V + (A_j - mean A).  The TMEM load is
            // warp-wide (.sync.aligned): every lane issues it, invalid rows included.
            wait(&bars->hd);
            if (!ok) break;
            const float *bh = bias + 3 * kH + 16 * q;
            float d[16];
            tmem_ld16(lane_t + rs, d);
            publish(&bars->hd_free);
            // epsilon-greedy (every quarter advances an identical copy of the
            // episode's LCG): u1 decides, the second state gives the random action
            const float u1 = lcg_uniform(s.rng);
            s.rng = s.rng * 1664525u + 1013904223u;
            const int a_rand = (int)(((uint64_t)(s.rng >> 8) * (uint64_t)kActions) >> 24);
            // this quarter's advantage sum (column order), first maximum and its
            // column, V (quarter 2) and A of the random action.  Q_j = V + (A_j -
            // mean A) is nondecreasing in A_j under float rounding, so the greedy
            // action is the first maximum of A and max Q = V + (max A - mean A).
            float sA = 0.f, mA = -INFINITY, Vq = 0.f, Ar = 0.f;
            int bA = 16 * q;
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const int j = 16 * q + k;
                const float A = d[k] + bh[k];
                if (j < kActions) {
                    sA += A;
                    if (A > mA) {
                        mA = A;
                        bA = j;
                    }
                    if (j == a_rand) Ar = A;
                } else if (j == kActions) {
                    Vq = A;
                }
            }
            if (q > 0) {
                hsum[(q - 1) * 128 + r] = sA;
                hqmax[(q - 1) * 128 + r] = mA;
                hbest[(q - 1) * 128 + r] = bA;
                if (q == 2) hval[r] = Vq;
                if (a_rand >= 16 * q && a_rand < 16 * q + 16) hqrand[r] = Ar;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->hx2[quad]);
                continue;
            }
            ok = warp_wait(&bars->hx2[quad], par, &abort_flag);
            if (!ok) break;
            const float meanA = ((sA + hsum[r]) + hsum[128 + r]) / (float)kActions;
            const float V = hval[r];
            // the first maximum over all 45 columns: a later quarter wins only if strictly greater
            int best = bA;
#pragma unroll
            for (int k = 0; k < 2; ++k)
                if (hqmax[k * 128 + r] > mA) {
                    mA = hqmax[k * 128 + r];
                    best = hbest[k * 128 + r];
                }
            if (a_rand >= 16) Ar = hqrand[r];
            const float qbest = V + (mA - meanA), q_rand = V + (Ar - meanA);
            const bool explore = u1 < a.epsilon;
            const int act = explore ? a_rand : best;
            const float q_sel = explore ? q_rand : qbest;
            const long long i = (long long)n * L + t;
            float v_in = 0.f, v_post = 0.f, rew = 0.f;
            int done = 0;
            if (valid) {
                v_in = s.V;
                float pnl;
                int label;
                env_trade(s, act, f[3], env, pnl, v_post, label, done);
                rew = env_window_reward(s, act, pnl, label, done, env);
            }
            // the next step's columns 48..55 (V and e after the trade), then the stores
            if (kRecycle) {
                // after a done, the next step starts at a fresh bar: one more LCG
                // state, over every bar that leaves room for the remaining steps
                long long nb = bar + 1;
                if (valid && done && t < L - 1) {
                    s.rng = s.rng * 1664525u + 1013904223u;
                    const uint64_t range = (uint64_t)(a.n_bars - L + t + 1);
                    nb = (long long)(((uint64_t)(s.rng >> 8) * range) >> 24);
                }
                if (n < a.N) a.bars[i] = valid ? (int32_t)bar : 0;
                if (nb != bar + 1) {
                    // this row's next state: the market columns of the new bar (the
                    // other quarters wrote the previous bar's), V = 1, e = 0
                    const float4 *src = reinterpret_cast<const float4 *>(a.Fpad + nb * kFPad);
#pragma unroll
                    for (int u = 0; u < 6; ++u) {
                        const float4 f0 = __ldg(src + 2 * u), f1 = __ldg(src + 2 * u + 1);
                        *reinterpret_cast<uint4 *>(X + sw128_offset(r, u)) =
                            make_uint4(pack_bf16x2(f0.x, f0.y), pack_bf16x2(f0.z, f0.w), pack_bf16x2(f1.x, f1.y),
                                       pack_bf16x2(f1.z, f1.w));
                    }
                    const float4 f12 = __ldg(src + 12);
                    float g[16] = {f12.x, f12.y, f12.z};
                    put_tail(g);
                } else {
                    put_tail(f);
                }
                bar_s[r] = (int)nb;
                rng_s[r] = s.rng;
                bar = nb;
                __syncwarp();
                if (lane == 0) mbar_arrive(&bars->ve);
            } else {
                put_tail(f);
            }
            publish(&bars->xt);
            if (n < a.N) {
                a.actions[i] = valid ? act : 0;
                a.dones[i] = done;
                a.rewards[i] = rew;
                a.v_in[i] = v_in;
                a.v_post[i] = v_post;
                a.q[i] = valid ? q_sel : 0.f;
            }
        }
    } else if (warp < kRMma) {
        // ------------------------------------------------------------ weight stream, stage st
        const int st = warp - kRProd0;
        if (lane == 0) {
            const long long total = (long long)kRUnitsPerStep * L + 1;
            long long last = -1;
            for (long long u = st; u < total; u += kStages) {
                const int i = rollout_unit(u);
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
            const uint32_t sX = smem_u32(X), sH = smem_u32(Hb), sRing = smem_u32(ring);
            long long g = 0;
            bool ok = true;
            // units are taken in stream order; each is released (its stage reusable
            // once the MMAs issued so far complete) when its MMAs are issued, the
            // next step's W1 only after the head
            auto take_at = [&](long long gg) -> uint32_t {
                const int st = (int)(gg % kStages);
                ok = ok && mbar_wait(&bars->full[st], (uint32_t)((gg / kStages) & 1), &abort_flag);
                tc_fence_after();
                return sRing + st * kStage;
            };
            auto release_at = [&](long long gg) { mma_commit(&bars->empty[gg % kStages]); };
            auto take = [&]() -> uint32_t { return take_at(g); };
            auto release = [&]() {
                release_at(g);
                ++g;
            };
            auto wait = [&](uint64_t *bar, uint32_t parity) {
                ok = ok && mbar_wait(bar, parity, &abort_flag);
                tc_fence_after();
            };
            auto chunk = [&](uint32_t col, uint32_t a_s, uint32_t b_s, uint32_t id, bool accumulate) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma<true>(tmem + col, desc_sw128(a_s + 32 * k), desc_sw128(b_s + 32 * k), id,
                              (accumulate || k > 0) ? 1u : 0u);
            };
            uint32_t u;
            u = take();
            wait(&bars->xm, 0);
            wait(&bars->xt, 0);
            if (ok) {
                chunk(0, sX, u, id256, false);
                release();
                mma_commit(&bars->q1);
            }
            for (int t = 0; t < L && ok; ++t) {
                const uint32_t par = t & 1, rs = par * 256, ro = 256 - rs;
                // layer 2 into the other region (the previous step's head was there)
                for (int c = 0; c < 4 && ok; ++c) {
                    u = take();
                    wait(&bars->h1[c], par);
                    if (c == 0 && t > 0) wait(&bars->hd_free, par ^ 1u);
                    if (!ok) break;
                    chunk(ro, sH + c * kChunk, u, id256, c > 0);
                    release();
                }
                if (!ok) break;
                mma_commit(&bars->q2);
                // layer 3 into region s
                for (int c = 0; c < 4 && ok; ++c) {
                    u = take();
                    wait(&bars->h2[c], par);
                    if (!ok) break;
                    chunk(rs, sH + c * kChunk, u, id256, c > 0);
                    release();
                }
                if (!ok) break;
                mma_commit(&bars->q3);
                // the next step's layer 1 into the other region (H2 is out of it): its
                // market columns (K16 steps 0-2) are in X already, written while
                // this step's layer 1 was drained, so they go in now and only the
                // portfolio columns wait for the environment step.  With recycling
                // a row's market columns change after the environment step: all of
                // layer 1 waits.
                const bool more = t + 1 < L;
                const long long g_w1 = g++;
                const uint32_t uw = take_at(g_w1);
                if (!ok) break;
                if (!kRecycle && more) {
                    wait(&bars->xm, par ^ 1u);
                    if (!ok) break;
#pragma unroll
                    for (int k = 0; k < 3; ++k)
                        mma<true>(tmem + ro, desc_sw128(sX + 32 * k), desc_sw128(uw + 32 * k), id256,
                                  k > 0 ? 1u : 0u);
                }
                // the head into [0, 48) of region s, K-chunk by K-chunk
                const long long g_hd = g++;
                u = take_at(g_hd);
                for (int c = 0; c < 4 && ok; ++c) {
                    wait(&bars->h3[c], par);
                    if (!ok) break;
                    chunk(rs, sH + c * kChunk, u + c * kHeadTile, id48, c > 0);
                }
                if (!ok) break;
                release_at(g_hd);
                mma_commit(&bars->hd);
                if (more) {
                    wait(&bars->xt, par ^ 1u);
                    if (kRecycle) wait(&bars->xm, par ^ 1u);
                    if (!ok) break;
                    if (kRecycle) chunk(ro, sX, uw, id256, false);
                    else mma<true>(tmem + ro, desc_sw128(sX + 96), desc_sw128(uw + 96), id256, 1u);
                    mma_commit(&bars->q1);
                }
                release_at(g_w1);
            }
            // every MMA issued has completed before TMEM is freed
            mma_commit(&bars->fin);
            mbar_wait_drain(&bars->fin, 0);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kRMma) {
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
    float *d_fpad = nullptr;   // the features with rows padded to kFPad floats, refilled every run
    cudaStream_t last_stream = nullptr;
    bool timing = false, timed_run = false;
    cudaEvent_t ev[4] = {};
    bool test_stall = false;   // dqn_test_stall: launch the target pass's stalling test build
    bool recycle = false;      // dqn_set_recycle: episode recycling
    int32_t *d_bars = nullptr; // recycling: the bar of every step [N L]
    size_t bars_cap = 0;
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
    cudaFree(h->d_bars);
    cudaFree(h->d_fpad);
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
        (e = cudaMalloc(&h->d_fpad, (size_t)dims->n_bars * kFPad * sizeof(float))) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_rollout_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_rollout_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kRSmem)) !=
            cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_target_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kTSmem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_target_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kTSmem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_target_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kTSmem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(dqn_target_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  kTSmem)) != cudaSuccess) {
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
    if (h->recycle && NL > h->bars_cap) {
        if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
        cudaFree(h->d_bars);
        h->d_bars = nullptr;
        h->bars_cap = 0;
        if ((e = cudaMalloc(&h->d_bars, NL * sizeof(int32_t))) != cudaSuccess) return cuda_fail(e, "cudaMalloc(bars)");
        h->bars_cap = NL;
    }
    int32_t *bars = h->recycle ? h->d_bars : nullptr;
    cudaStream_t s = (cudaStream_t)stream;
    h->last_stream = s;
    const rollout_dims &d = h->dims;
    if ((e = cudaMemsetAsync(h->d_status, 0, sizeof(int), s)) != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    const EnvConst env{d.barrier, d.max_hold, d.pt_scale, d.sl_scale, d.div_window, d.div_thresh, d.div_penalty,
                       d.cur_coef, d.risk_coef, d.tx_base, d.spread, h->d_div};
    const RolloutArgs ra{features, h->d_fpad, starts, seeds, N, L, d.n_bars, epsilon, actions, dones, rewards, td,
                         h->d_vpost, q, h->d_status, env, bars};
    auto mark = [&](int i) { return h->timing ? cudaEventRecord(h->ev[i], s) : cudaSuccess; };
    if ((e = launch_pad_features(features, h->d_fpad, d.n_bars, s)) != cudaSuccess)
        return cuda_fail(e, "feature padding launch");
    if ((e = mark(0)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    if (h->recycle) dqn_rollout_kernel<true><<<(N + 127) / 128, kRThreads, kRSmem, s>>>(ra, h->img);
    else dqn_rollout_kernel<false><<<(N + 127) / 128, kRThreads, kRSmem, s>>>(ra, h->img);
    if ((e = cudaGetLastError()) != cudaSuccess) return cuda_fail(e, "DQN rollout launch");
    if ((e = mark(1)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    const StatesArgs sa{features, starts, N, L, d.n_bars, actions, dones, td, d.spread, states, h->d_fpad, bars};
    if ((e = launch_states(sa, s)) != cudaSuccess) return cuda_fail(e, "state-row launch");
    if ((e = mark(2)) != cudaSuccess) return cuda_fail(e, "cudaEventRecord");
    const TargetArgs ta{features, h->d_fpad, starts, N, L, d.n_bars, gamma, actions, dones, rewards, td, h->d_vpost,
                        q, next_states, h->d_status, env, bars};
    const long long tiles = (long long)((NL + 127) / 128);
    const int grid = (int)(tiles < h->sms ? tiles : h->sms);
    if (h->test_stall) {
        if (h->recycle) dqn_target_kernel<true, true><<<grid, kTThreads, kTSmem, s>>>(ta, h->img);
        else dqn_target_kernel<true, false><<<grid, kTThreads, kTSmem, s>>>(ta, h->img);
    } else {
        if (h->recycle) dqn_target_kernel<false, true><<<grid, kTThreads, kTSmem, s>>>(ta, h->img);
        else dqn_target_kernel<false, false><<<grid, kTThreads, kTSmem, s>>>(ta, h->img);
    }
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

int dqn_set_recycle(dqn_handle *h, int on)
{
    clear_error();
    if (!h) return set_error(ROLLOUT_ERR_INVALID, "null handle");
    h->recycle = on != 0;
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
