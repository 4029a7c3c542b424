// value_umma.cu -- tensor-core value phase (phase 2), bf16 operands, critic
// 54->512->384->256->128->64->1 and curiosity (54+45)->64->54.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A step 5 (critic) and step 9 (curiosity
// forward model; bonus = cur_coef * MSE against the pre-reset next state);
// section "Weight Layout".
//
// The critic and the curiosity model do not feed the state trajectory, so they
// run here over every tuple at once instead of inside the serial step loop.
// A persistent CTA takes tiles of 128 consecutive rows (tuples, then one
// bootstrap row per episode: the pre-reset next state after the last step) and
// runs every layer as M=128 tcgen05 MMAs with f32 accumulators in TMEM.
//
// Warp roles (20 warps):
//   0-15  row warps: warp w serves TMEM lanes / rows 32*(w%4)..+31 and the
//         column quarter w/4 of every 64-column chunk.  They build the state
//         rows (A operand), drain TMEM chunk by chunk (bias, ReLU, bf16
//         rounding) into the next layer's swizzled A operand, and finish with
//         the head dot product, the curiosity MSE and the stores.  The next
//         tile's row metadata is loaded one tile ahead.
//   16-18 producers: stream the weights (pre-swizzled on the host, grouped
//         into 26 units of <= 32 KB per tile) from L2 with 1-D bulk TMA into a
//         three-stage ring.  Producer s owns stage s and so waits on its empty
//         barrier strictly in order; the bulk copies of one warp complete one
//         after another, those of different warps overlap.
//         (lane 1 of warp 16 stages each tile's market-feature rows)
//   19    allocates TMEM; one lane issues the MMAs and commits
//
// Per tile the MMA lane runs (TMEM columns in brackets):
//   CUR1 [320,384) = X C1^T and D1_0 [384,512) = X W1[rows 0..127]^T, one
//   N=192 MMA (the previous tile's layer 3 has left [256,512))
//   CUR2 [256,320) = Z C2^T                        (after the rows wrote Z)
//   for i < 8:  D2 [0,384) += h1_i W2[:, chunk i]^T  (after rows wrote h1_i;
//                 for i = 0 the columns [256,384) also wait for CUR2's drain)
//     odd i < 7, first: D1_c = X W1[rows 128c..]^T, c = (i+1)/2, into the
//                 buffer the rows just emptied (h1_{i-1}, h1_i came from it)
//   D3 [256,512) += h2_k W3^T, k = 4,5,0,1,2,3       (as the rows write h2_k)
//   D4 [0,128)   += h3_k W4^T, k = 0..3
//   D5 [128,192) += h4_k W5^T, k = 0..1
// so layer 1 never exists whole (its 128-column chunks are produced while the
// tensor pipe accumulates layer 2: N=128 MMAs cost the tensor pipe about what
// N=64 ones do, so four of them replace eight) and every later layer starts on
// its first K-chunk while the rows still drain the rest of the previous one.
// A layer-1 chunk is issued ahead of layer 2's MMAs on h1 slot 1, so the rows
// drain its second half into slot 1 only after a commit (acc_h1free) shows
// that those MMAs are done.  The rows
// build X and Z of the next tile at the end of the current one, and at the
// start of a tile drain h1_0 before the curiosity error, so that layer 2
// starts without waiting for the curiosity epilogues.
// Shared-memory operand slots (128 rows x 128 B each): X -> 2, Z -> 3,
// h1 chunks -> 0/1 (alternating), h2 -> 0..5, h3 -> 0..3, h4 -> 0..1.  From
// the end of layer 3 of the previous tile until the curiosity epilogue, slots
// 4-5 hold the tile's market-feature rows: one bulk copy per episode the tile
// touches (at most four), each a run of consecutive bars of the feature
// matrix, so that X and the curiosity targets are built from shared memory
// instead of gathering 204-byte rows thread by thread.
// Every handoff has its own mbarrier (one phase per tile) so that no barrier
// can complete twice before its waiter has seen the first completion.
#include "env.cuh"
#include "umma.cuh"
#include "umma_path.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kRowWarps = 16;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kProducers = 3;            // one per ring stage
constexpr int kProdWarp0 = kRowWarps, kMmaWarp = kRowWarps + kProducers;
constexpr int kThreads = (kMmaWarp + 1) * 32;
constexpr int kSlot = 128 * 128;
constexpr int kNumSlots = 6;
constexpr int kStage = 32 * 1024;
constexpr int kStages = kProducers;
constexpr int kUnits = 26;
constexpr int kXSlot = 2, kZSlot = 3, kFeatSlot = 4;
constexpr int kFeatFloats = 2 * kSlot / 4;      // feature staging area (slots 4-5): 8192 floats
constexpr int kMaxSeg = 4;                      // episodes of one tile staged at most
constexpr int kBiasFloats = 1600;
constexpr int kOneHotLd = kCurH + 4;             // padded row: the rows of different actions start on different banks
constexpr int kOneHotFloats = kActions * kOneHotLd;
constexpr int kSmem = kNumSlots * kSlot + kStages * kStage + (kBiasFloats + kOneHotFloats) * 4 + 2 * 4 * 128 * 4 + 1024;
static_assert(kSmem <= 232448, "value kernel shared memory");

// bias block layout in shared memory (floats)
constexpr int kB1 = 0, kB2 = 512, kB3 = 896, kB4 = 1152, kB5 = 1280, kHW = 1344, kHB = 1408, kC1B = 1412,
              kC2B = 1476;

// TMEM columns
constexpr uint32_t kColCur1 = 320, kColCur2 = 256, kColD1 = 384, kColD2 = 0, kColD3 = 256, kColD4 = 0, kColD5 = 128;

struct Bars {
    uint64_t full[kStages], empty[kStages];
    uint64_t act_x, act_z, act_cz, act_h1[2], act_h2[6], act_h3[4], act_h4[2];   // act_cz: CUR2 columns drained
    uint64_t acc_cur, acc_d1, acc_h1free, acc_main, final_;   // acc_h1free: h1 slot 1 read
    uint64_t feat_full;        // the staged feature rows of the next tile have landed
    uint64_t feat_free;        // layer 3 has read slots 4-5: the next tile's rows may be staged there
};

// Where the feature rows of a tile's episodes sit in the staging area.
// Segment j covers episode n0 + j: bars [lo, hi) of the feature matrix at
// float offset soff; lo < 0 when the episode is not staged.
struct SegTable {
    long long n0;
    int count;
    int lo[kMaxSeg], hi[kMaxSeg], soff[kMaxSeg];
};

// the starts of the (up to kMaxSeg) episodes of the tile at r0, loaded early
struct SegPre {
    long long r0, n0;
    int count;
    int st[kMaxSeg];
};

__device__ __forceinline__ float bf16_round(float x) { return __uint_as_float(pack_bf16x2(0.f, x) & 0xFFFF0000u); }

// x / L for x >= 0, in 32 bits when x fits (the 64-bit division is a long
// instruction sequence)
__device__ __forceinline__ long long div_L(long long x, int L)
{
    return x <= 0x7fffffffLL ? (long long)((uint32_t)x / (uint32_t)L) : x / L;
}

__device__ __forceinline__ void seg_prefetch(const ValueArgs &a, long long r0, SegPre &p)
{
    const long long NL = (long long)a.N * a.L;
    p.r0 = r0;
    p.n0 = 0;
    p.count = 0;
    if (r0 < NL) {
        p.n0 = div_L(r0, a.L);
        const long long r_end = r0 + 128 < NL ? r0 + 128 : NL;
        const long long n_last = div_L(r_end - 1, a.L);
        p.count = (int)(n_last - p.n0 + 1 < kMaxSeg ? n_last - p.n0 + 1 : kMaxSeg);
    }
#pragma unroll
    for (int j = 0; j < kMaxSeg; ++j) {
        const long long n = p.n0 + j < a.N ? p.n0 + j : a.N - 1;
        p.st[j] = __ldg(a.starts + n);
    }
}

// One thread: lays the segments out, publishes the table and issues the
// copies, completing `bar` with their bytes.  A segment starts on a bar that
// is a multiple of 4 and spans a multiple of 4 bars (4 x 204 bytes = 816, a
// multiple of 16, as a bulk copy requires); it covers the bars of the tile's
// steps plus the next bar (the curiosity target) and never reaches past the
// feature matrix.  Rows outside every segment are read from global memory.
__device__ __forceinline__ void seg_issue(const ValueArgs &a, const SegPre &p, SegTable &T, float *area,
                                          uint64_t *bar)
{
    const long long NL = (long long)a.N * a.L;
    const long long r_end = p.r0 + 128 < NL ? p.r0 + 128 : NL;
    int soff = 0;
    uint32_t total = 0;
    T.n0 = p.n0;
    T.count = p.count;
#pragma unroll
    for (int j = 0; j < kMaxSeg; ++j) {
        T.lo[j] = -1;
        T.hi[j] = -1;
        T.soff[j] = 0;
        if (j >= p.count) continue;
        const long long n = p.n0 + j, e0 = n * a.L;
        const int ta = (int)((p.r0 > e0 ? p.r0 : e0) - e0);
        const int tb = (int)((r_end < e0 + a.L ? r_end : e0 + a.L) - 1 - e0);
        const int st = p.st[j];
        if (!start_ok(st, a.L, a.n_bars)) continue;
        const long long lo = ((long long)st + ta) & ~3LL;
        long long hi = ((long long)st + tb + 2 + 3) & ~3LL;
        if (hi > a.n_bars) hi = lo + (((long long)a.n_bars - lo) & ~3LL);
        const int nb = (int)(hi - lo);
        if (nb <= 0 || soff + nb * kMarket > kFeatFloats) continue;
        T.lo[j] = (int)lo;
        T.hi[j] = (int)hi;
        T.soff[j] = soff;
        soff += nb * kMarket;
        total += (uint32_t)nb * kMarket * 4u;
    }
    mbar_arrive_expect_tx(bar, total);
#pragma unroll
    for (int j = 0; j < kMaxSeg; ++j)
        if (T.lo[j] >= 0)
            bulk_g2s(area + T.soff[j], a.F + (long long)T.lo[j] * kMarket,
                     (uint32_t)(T.hi[j] - T.lo[j]) * kMarket * 4u, bar);
}

// float offset of bar `b` of episode n in the staging area, or -1
__device__ __forceinline__ int staged_off(const SegTable &T, long long n, long long b)
{
    const long long j = n - T.n0;
    if (j < 0 || j >= T.count) return -1;
    const int lo = T.lo[j];
    if (lo < 0 || b < lo || b >= T.hi[j]) return -1;
    return T.soff[j] + (int)(b - lo) * kMarket;
}

struct RowInfo {
    int kind;            // 0 tuple, 1 bootstrap row, 2 tuple of an invalid episode, 3 bootstrap of one, -1 none
    int n;               // episode
    long long row;       // flat tuple index (kind 0/2) or the slot receiving the bootstrap value (kind 1/3)
    int bar;             // bar of the state row (< n_bars)
    int act;
    float vin, ein, vpost, rew;
};

// Per-row metadata, loaded one tile ahead: every load's address depends only
// on the row index (issued at the start of the previous tile, consumed in its
// middle), so no thread stalls on them.
struct RowFetch {
    long long r, row;          // flat row, tuple index / bootstrap slot
    int n, t, is_boot;         // episode, step, bootstrap row?
    int start, act, aprev, dprev;
    float vin, vpost, rew;
};

__device__ __forceinline__ void issue_meta(const ValueArgs &a, long long r, RowFetch &f)
{
    const long long NL = (long long)a.N * a.L;
    const int L = a.L;
    f.r = r;
    f.is_boot = r >= NL;
    const long long rc = r < NL + a.N ? r : NL + a.N - 1;      // rows past the end read row `total-1`
    if (f.is_boot) {
        f.n = (int)(rc - NL);
        f.t = L - 1;
    } else {
        f.n = (int)div_L(rc, L);
        f.t = (int)(rc - (long long)f.n * L);
    }
    f.row = (long long)f.n * L + f.t;
    const long long prev = f.t > 0 ? f.row - 1 : f.row;
    f.start = __ldg(a.starts + f.n);
    f.act = a.actions[f.row];
    f.vin = f.is_boot ? a.v_post[f.row] : a.values[f.row];
    f.vpost = a.v_post[f.row];
    f.rew = a.rewards[f.row];                  // base reward: the curiosity bonus is added to it
    f.aprev = a.actions[prev];
    f.dprev = a.dones[prev];
}

__device__ __forceinline__ RowInfo resolve(const ValueArgs &a, const RowFetch &f)
{
    RowInfo ri{};
    const long long NL = (long long)a.N * a.L;
    const bool ok = start_ok(f.start, a.L, a.n_bars);
    ri.n = f.n;
    ri.row = f.row;
    ri.act = f.act;
    ri.rew = f.rew;
    if (f.r >= NL + a.N) {
        ri.kind = -1;
    } else if (!f.is_boot) {
        ri.kind = ok ? 0 : 2;
        ri.bar = f.start + f.t;
        ri.vin = f.vin;
        ri.vpost = f.vpost;
        ri.ein = (f.t == 0 || f.dprev) ? 0.f : exposure_of(f.aprev);
    } else {
        ri.kind = ok ? 1 : 3;
        ri.bar = f.start + a.L;
        ri.vin = f.vin;
        ri.ein = exposure_of(f.act);
    }
    if (ri.kind != 0 && ri.kind != 1) ri.bar = 0;
    return ri;
}

// state columns [16q, 16q+16) of the row: [F[bar], V, e, spread, 0...]
__device__ __forceinline__ void state_cols(const ValueArgs &a, const RowInfo &ri, const SegTable &T,
                                           const float *area, int q, float (&xv)[16])
{
    const bool has = ri.kind == 0 || ri.kind == 1;
    const int off = ri.kind == 0 ? staged_off(T, ri.n, ri.bar) : -1;
    const float *src = off >= 0 ? area + off : a.F + (long long)ri.bar * kMarket;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int c = 16 * q + j;
        float x = 0.f;
        if (has) {
            if (c < kMarket) x = src[c];
            else if (c == kMarket) x = ri.vin;
            else if (c == kMarket + 1) x = ri.ein;
            else if (c == kMarket + 2) x = a.env.spread;
        }
        xv[j] = x;
    }
}

// curiosity target columns [16q, 16q+16): the pre-reset next state
// [F[bar+1], V', e', spread] (used for tuples only)
__device__ __forceinline__ void target_cols(const ValueArgs &a, const RowInfo &ri, const SegTable &T,
                                            const float *area, int q, float (&tv)[16])
{
    const int off = ri.kind == 0 ? staged_off(T, ri.n, ri.bar + 1) : -1;
    const float *src = off >= 0 ? area + off : a.F + (ri.kind == 0 ? (long long)ri.bar + 1 : 0LL) * kMarket;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int c = 16 * q + j;
        float x = 0.f;
        if (c < kMarket) x = ri.kind == 0 ? src[c] : 0.f;
        else if (c == kMarket) x = ri.vpost;
        else if (c == kMarket + 1) x = exposure_of(ri.act);
        else if (c == kMarket + 2) x = a.env.spread;
        tv[j] = x;
    }
}

// 16 f32 values -> 2 bf16 units of row r, columns [16q, 16q+16) of operand tile
// `tile`; D: also the rounded values of columns below n_valid to dst (test hook)
template <bool D = false>
__device__ __forceinline__ void put16(uint8_t *tile, int r, int q, const float (&v)[16], float *dst = nullptr,
                                      int n_valid = 0)
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 p;
        p.x = pack_bf16x2(v[8 * h + 0], v[8 * h + 1]);
        p.y = pack_bf16x2(v[8 * h + 2], v[8 * h + 3]);
        p.z = pack_bf16x2(v[8 * h + 4], v[8 * h + 5]);
        p.w = pack_bf16x2(v[8 * h + 6], v[8 * h + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 2 * q + h)) = p;
        if constexpr (D) {
            if (dst) {
                const uint32_t w4[4] = {p.x, p.y, p.z, p.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = unpack_bf16x2(w4[k]);
                    const int c = 16 * q + 8 * h + 2 * k;
                    if (c < n_valid) dst[8 * h + 2 * k] = f.x;
                    if (c + 1 < n_valid) dst[8 * h + 2 * k + 1] = f.y;
                }
            }
        }
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

// 16 f32 values -> relu -> 2 bf16 units, as put16; D: also the rounded
// values to dst[0..16) when dst is not null (test hook)
template <bool D = false>
__device__ __forceinline__ void put16_relu(uint8_t *tile, int r, int q, const float (&v)[16], float *dst = nullptr)
{
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        uint4 p;
        p.x = pack_bf16x2_relu(v[8 * h + 0], v[8 * h + 1]);
        p.y = pack_bf16x2_relu(v[8 * h + 2], v[8 * h + 3]);
        p.z = pack_bf16x2_relu(v[8 * h + 4], v[8 * h + 5]);
        p.w = pack_bf16x2_relu(v[8 * h + 6], v[8 * h + 7]);
        *reinterpret_cast<uint4 *>(tile + sw128_offset(r, 2 * q + h)) = p;
        if constexpr (D) {
            if (dst) {
                const float2 a = unpack_bf16x2(p.x), b = unpack_bf16x2(p.y), c = unpack_bf16x2(p.z),
                             d = unpack_bf16x2(p.w);
                reinterpret_cast<float4 *>(dst + 8 * h)[0] = make_float4(a.x, a.y, b.x, b.y);
                reinterpret_cast<float4 *>(dst + 8 * h)[1] = make_float4(c.x, c.y, d.x, d.y);
            }
        }
    }
}

// the test hook's row of a tile row (ActDump), or nullptr
__device__ __forceinline__ float *dump_row(const ValueArgs &a, const RowInfo &ri)
{
    if (ri.kind == 0) return a.dump.row(ri.n, (int)(ri.row - (long long)ri.n * a.L), a.L);
    if (ri.kind == 1) return a.dump.row(ri.n, a.L, a.L);
    return nullptr;
}

// relu(D[cols] + bias) rounded to bf16 into row r / quarter q of operand tile
// `tile` (D: and to dst[0..16) when dst is not null)
template <bool D = false>
__device__ __forceinline__ void drain16(uint32_t taddr, const float *bias, uint8_t *tile, int r, int q,
                                        float *dst = nullptr)
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
    put16_relu<D>(tile, r, q, v, dst);
}

__device__ __forceinline__ void row_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kRowThreads) : "memory"); }

// row_sync that also returns the AND of `pred` over every row thread, so that
// all row warps leave the tile loop on the same tile
__device__ __forceinline__ bool row_sync_and(bool pred)
{
    uint32_t out;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.and.pred q, 1, %2, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(out)
        : "r"((uint32_t)pred), "n"(kRowThreads)
        : "memory");
    return out != 0;
}

// one arrival per warp, after every lane's generic-proxy smem accesses and
// TMEM reads: each lane fences its own accesses, the warp synchronises, lane
// 0 arrives (512 per-thread arrivals on one barrier would serialise in the
// shared-memory atomic unit)
__device__ __forceinline__ void publish(uint64_t *bar)
{
    fence_async_smem();
    tc_fence_before();
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

struct MmaCtx {
    uint32_t tmem, s_slots;
    volatile int *abort;
    bool ok;
    __device__ __forceinline__ uint32_t slot(int s) const { return s_slots + s * kSlot; }
    // D[col] (+)= A[a] * B[b]^T over one 128-byte K-chunk, N = n
    __device__ __forceinline__ void mma_chunk(uint32_t col, uint32_t a, uint32_t b, int n, bool accumulate) const
    {
        const uint32_t id = idesc(true, 128, n);
#pragma unroll
        for (int k = 0; k < 4; ++k)
            mma<true>(tmem + col, desc_sw128(a + 32 * k), desc_sw128(b + 32 * k), id,
                      (accumulate || k > 0) ? 1u : 0u);
    }
    __device__ __forceinline__ void wait(uint64_t *bar, uint32_t &phase)
    {
        ok = ok && mbar_wait(bar, phase, abort);
        phase ^= 1u;
        tc_fence_after();
    }
};

// kStall: a test build in which the first producer of CTA 0 issues no copy, so
// that CTA's MMA issuer waits on a weight stage that never fills and the
// bounded-wait exit runs (rollout_test_stall).  kDump: a test build that also
// writes every row's rounded hidden activations (rollout_test_activations).
template <bool kStall, bool kDump>
__global__ void __launch_bounds__(kThreads, 1) value_umma_bf16_kernel(ValueArgs a, UmmaWeights w)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *slots = sm;
    uint8_t *ring = sm + kNumSlots * kSlot;
    float *bias = reinterpret_cast<float *>(ring + kStages * kStage);
    float *onehot = bias + kBiasFloats;                  // curiosity layer-1 one-hot columns [45][kOneHotLd]
    float *part = onehot + kOneHotFloats;                // [2][4][128] partial sums
    float *feat = reinterpret_cast<float *>(slots + kFeatSlot * kSlot);
    __shared__ __align__(8) Bars B;
    __shared__ SegTable seg;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) {
        abort_sh = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&B.full[s], 1);
            mbar_init(&B.empty[s], 1);
        }
        mbar_init(&B.act_x, kRowWarps);
        mbar_init(&B.act_z, kRowWarps);
        mbar_init(&B.act_cz, kRowWarps);
        for (int i = 0; i < 2; ++i) mbar_init(&B.act_h1[i], kRowWarps);
        for (int i = 0; i < 6; ++i) mbar_init(&B.act_h2[i], kRowWarps);
        for (int i = 0; i < 4; ++i) mbar_init(&B.act_h3[i], kRowWarps);
        for (int i = 0; i < 2; ++i) mbar_init(&B.act_h4[i], kRowWarps);
        mbar_init(&B.acc_cur, 1);
        mbar_init(&B.acc_d1, 1);
        mbar_init(&B.acc_h1free, 1);
        mbar_init(&B.acc_main, 1);
        mbar_init(&B.final_, 1);
        mbar_init(&B.feat_full, 1);
        mbar_init(&B.feat_free, 1);
        fence_mbar_init();
    }
    // biases, head weights and one-hot columns (f32; the latter two already bf16-rounded)
    {
        const float *vec = w.vec;
        for (int i = tid; i < kBiasFloats; i += kThreads) {
            float v = 0.f;
            if (i < kB2) v = vec[w.job[kJobCrit1].bias_off + i];
            else if (i < kB3) v = vec[w.job[kJobCrit2].bias_off + i - kB2];
            else if (i < kB4) v = vec[w.job[kJobCrit3].bias_off + i - kB3];
            else if (i < kB5) v = vec[w.job[kJobCrit4].bias_off + i - kB4];
            else if (i < kHW) v = vec[w.job[kJobCrit5].bias_off + i - kB5];
            else if (i < kHB) v = vec[w.head_w_off + i - kHW];
            else if (i == kHB) v = vec[w.head_b_off];
            else if (i >= kC1B && i < kC2B) v = vec[w.job[kJobCur1].bias_off + i - kC1B];
            else if (i >= kC2B && i < kC2B + 64) v = vec[w.job[kJobCur2].bias_off + i - kC2B];
            bias[i] = v;
        }
        for (int i = tid; i < kActions * kCurH; i += kThreads)
            onehot[(i / kCurH) * kOneHotLd + i % kCurH] = vec[w.onehot_off + i];
    }
    if (warp == kMmaWarp) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int *abort = &abort_sh;

    const long long total = (long long)a.N * a.L + a.N;
    const long long n_tiles = (total + 127) / 128;

    if (warp >= kProdWarp0 && warp < kMmaWarp) {
        // ------------------------------------------------------------ producers
        const int ps = warp - kProdWarp0;             // the ring stage this warp fills
        if (lane == 0) {
            uint32_t k = 0;                            // uses of stage ps so far
            long long g = 0;                           // unit counter over all tiles: unit g goes to stage g % kStages
            bool ok = true;
            const bool silent = kStall && blockIdx.x == 0 && ps == 0;
            for (long long tile = blockIdx.x; tile < n_tiles && ok && !silent; tile += gridDim.x) {
                for (int u = 0; u < kUnits && ok; ++u, ++g) {
                    if (g % kStages != ps) continue;
                    const uint32_t bytes = w.unit_bytes[u];
                    ok = mbar_wait(&B.empty[ps], (k & 1u) ^ 1u, abort);   // release of the previous use
                    if (!ok) break;
                    mbar_arrive_expect_tx(&B.full[ps], bytes);
                    bulk_g2s(ring + ps * kStage, w.stream + w.unit_off[u], bytes, &B.full[ps]);
                    ++k;
                }
            }
            // the last copy into this stage has landed once the MMA lane has released it
            if (ok && k > 0) ok = mbar_wait(&B.empty[ps], (k - 1) & 1u, abort);
            if (!ok) {   // aborted: give copies already issued time to land (bounded)
                const long long c0 = clock64();
                while (clock64() - c0 < 4000000) { }
            }
        } else if (ps == 0 && lane == 1) {
            // ---- feature stager (lane 1 of the first producer warp): stages each
            // tile's market-feature rows into slots 4-5, for the first tile at once,
            // for every later one once the rows report that layer 3 of the previous
            // tile has read those slots; loading the episode starts here keeps
            // their latency off the row warps
            bool ok = true;
            uint32_t ph = 0, issued = 0;
            for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                SegPre pre;
                seg_prefetch(a, tile * 128, pre);
                if (tile != blockIdx.x) {
                    ok = mbar_wait(&B.feat_free, ph, abort);
                    ph ^= 1u;
                    if (!ok) break;
                }
                seg_issue(a, pre, seg, feat, &B.feat_full);
                ++issued;
            }
            // the last copies have landed before the CTA may exit, also after an
            // abort (bounded wait independent of the abort flag)
            int never = 0;
            if (issued > 0) mbar_wait(&B.feat_full, (issued - 1) & 1u, &never, 100000000ull);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            MmaCtx m{tmem, smem_u32(slots), abort, true};
            const uint32_t s_ring = smem_u32(ring);
            int stage = 0;
            uint32_t ring_ph = 0;
            uint32_t ph_x = 0, ph_z = 0, ph_cz = 0, ph_h1[2] = {0, 0}, ph_h2[6] = {}, ph_h3[4] = {}, ph_h4[2] = {};
            auto take = [&]() -> uint32_t {      // wait for the next weight unit
                uint32_t p = ring_ph;
                m.wait(&B.full[stage], p);
                return s_ring + stage * kStage;
            };
            auto release = [&]() {               // stage reusable once these MMAs complete
                mma_commit(&B.empty[stage]);
                if (++stage == kStages) { stage = 0; ring_ph ^= 1u; }
            };
            for (long long tile = blockIdx.x; tile < n_tiles && m.ok; tile += gridDim.x) {
                // ---- unit 0: CUR1 and D1_0 as one N=192 MMA (C1's 64 rows and W1's
                // first 128 are contiguous in the unit, CUR1's columns [320,384)
                // adjoin D1's), then CUR2
                m.wait(&B.act_x, ph_x);
                uint32_t u = take();
                m.mma_chunk(kColCur1, m.slot(kXSlot), u, 192, false);
                mma_commit(&B.acc_cur);
                mma_commit(&B.acc_d1);
                m.wait(&B.act_z, ph_z);
                m.mma_chunk(kColCur2, m.slot(kZSlot), u + 24576, 64, false);
                mma_commit(&B.acc_cur);
                release();
                // ---- layer 2 over the h1 chunks (two units per K-chunk): K-chunk 0 takes
                // rows 0-255 of W2 first (the rest waits for CUR2's drain); every later
                // one takes rows 256-383 first, for odd i preceded by the next layer-1 chunk
                u = take();
                m.wait(&B.act_h1[0], ph_h1[0]);
                m.mma_chunk(kColD2, m.slot(0), u, 256, false);
                release();
                u = take();
                m.wait(&B.act_cz, ph_cz);                      // D2 columns [256,384) begin where CUR2 was
                m.mma_chunk(kColD2 + 256, m.slot(0), u, 128, false);
                release();
                for (int i = 1; i < 8; ++i) {
                    const bool d1 = (i & 1) && i < 7;
                    u = take();
                    m.wait(&B.act_h1[i & 1], ph_h1[i & 1]);
                    if (d1) {                                   // the rows have emptied the layer-1 buffer
                        m.mma_chunk(kColD1, m.slot(kXSlot), u, 128, false);
                        mma_commit(&B.acc_d1);
                    }
                    m.mma_chunk(kColD2 + 256, m.slot(i & 1), u + (d1 ? 16384 : 0), 128, true);
                    release();
                    u = take();
                    m.mma_chunk(kColD2, m.slot(i & 1), u, 256, true);
                    if (d1) mma_commit(&B.acc_h1free);         // h1 slot 1 may take the next chunk
                    release();
                }
                mma_commit(&B.acc_main);
                // ---- layer 3, K-chunks in the order the rows release them
                for (int kk = 0; kk < 6; ++kk) {
                    const int k = kk < 2 ? 4 + kk : kk - 2;
                    u = take();
                    m.wait(&B.act_h2[k], ph_h2[k]);
                    m.mma_chunk(kColD3, m.slot(k), u, 256, kk > 0);
                    release();
                }
                mma_commit(&B.acc_main);
                // ---- layer 4 (two units of two K-chunks)
                for (int h = 0; h < 2; ++h) {
                    u = take();
                    for (int k = 2 * h; k < 2 * h + 2; ++k) {
                        m.wait(&B.act_h3[k], ph_h3[k]);
                        m.mma_chunk(kColD4, m.slot(k), u + 16384 * (k - 2 * h), 128, k > 0);
                    }
                    if (h == 1) mma_commit(&B.acc_main);
                    release();
                }
                // ---- layer 5
                u = take();
                for (int k = 0; k < 2; ++k) {
                    m.wait(&B.act_h4[k], ph_h4[k]);
                    m.mma_chunk(kColD5, m.slot(k), u + 8192 * k, 64, k > 0);
                }
                mma_commit(&B.acc_main);
                release();
            }
            // every MMA issued must complete before TMEM is released (bounded wait)
            mma_commit(&B.final_);
            int never = 0;
            mbar_wait(&B.final_, 0, &never, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ row warps
        const int r = 32 * (warp & 3) + lane;                 // operand row / TMEM lane
        const int q = warp >> 2;                               // column quarter of every 64-col chunk
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 16 * q;
        uint32_t ph_cur = 0, ph_d1 = 0, ph_free = 0, ph_main = 0, ph_feat = 0;
        bool ok = true;
        auto wait_acc = [&](uint64_t *bar, uint32_t &phase) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(bar, phase, abort));
            phase ^= 1u;
            tc_fence_after();
        };
        float *part_v = part, *part_s = part + 4 * 128;
        auto build_x = [&](const RowInfo &ri) {
            ok = __all_sync(0xffffffffu, ok && mbar_wait(&B.feat_full, ph_feat, abort));
            ph_feat ^= 1u;
            float xv[16];
            state_cols(a, ri, seg, feat, q, xv);
            float *dx = nullptr;
            if constexpr (kDump) {
                dx = dump_row(a, ri);
                if (dx) dx += 16 * q;
            }
            put16<kDump>(slots + kXSlot * kSlot, r, q, xv, dx, kState);
            publish(&B.act_x);
        };

        // curiosity layer 1 of a tile: state part from TMEM, one-hot column gathered -> Z
        auto cur1_epilogue = [&](const RowInfo &ri) {
            wait_acc(&B.acc_cur, ph_cur);
            float v[16];
            tmem_ld16(lane_addr + kColCur1, v);
            const int act = (ri.act >= 0 && ri.act < kActions) ? ri.act : 0;
            const float4 *oh = reinterpret_cast<const float4 *>(onehot + act * kOneHotLd + 16 * q);
            const float4 *b4 = reinterpret_cast<const float4 *>(bias + kC1B + 16 * q);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 o = oh[k], b = b4[k];
                v[4 * k + 0] = (v[4 * k + 0] + o.x) + b.x;
                v[4 * k + 1] = (v[4 * k + 1] + o.y) + b.y;
                v[4 * k + 2] = (v[4 * k + 2] + o.z) + b.z;
                v[4 * k + 3] = (v[4 * k + 3] + o.w) + b.w;
            }
            float *dz = nullptr;
            if constexpr (kDump) {
                dz = dump_row(a, ri);
                if (dz && ri.kind == 0) dz += a.dump.cur_off + 16 * q;
                else dz = nullptr;
            }
            put16_relu<kDump>(slots + kZSlot * kSlot, r, q, v, dz);
            publish(&B.act_z);
        };

        long long tile = blockIdx.x;
        RowFetch nf;
        issue_meta(a, tile * 128 + r, nf);
        RowInfo nri = resolve(a, nf);
        build_x(nri);
        cur1_epilogue(nri);
        // a wait that expired in one row warp may have succeeded in another (the
        // barrier completing just after the limit): agree before the first
        // row_sync, so that every row warp runs the same barriers
        ok = row_sync_and(ok);

        for (; tile < n_tiles && ok; tile += gridDim.x) {
            const RowInfo ri = nri;
            const long long next = tile + gridDim.x;
            const bool has_next = next < n_tiles;
            float *drow = nullptr;                              // test hook: this row's activation dump
            if constexpr (kDump) drow = dump_row(a, ri);
            // column c of critic hidden layer l in the dump row, or nullptr
            auto dcol = [&](int l, int c) -> float * { return drow ? drow + a.dump.crit_off[l] + c : nullptr; };
            // ---- h1 chunk 0 first: the tensor pipe waits for it
            wait_acc(&B.acc_d1, ph_d1);
            drain16<kDump>(lane_addr + kColD1, bias + kB1 + 16 * q, slots, r, q, dcol(0, 16 * q));
            publish(&B.act_h1[0]);
            // ---- curiosity layer 2: squared error against the pre-reset next state
            wait_acc(&B.acc_cur, ph_cur);
            {
                float tv[16];
                target_cols(a, ri, seg, feat, q, tv);
                float v[16];
                tmem_ld16(lane_addr + kColCur2, v);
                float se = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    if (16 * q + j < kState) {
                        const float d = (v[j] + bias[kC2B + 16 * q + j]) - tv[j];
                        se = fmaf(d, d, se);
                    }
                }
                part_s[q * 128 + r] = se;
                publish(&B.act_cz);                            // its TMEM columns are layer 2's next
            }
            // ---- h1 chunks 1..7 (the tensor pipe accumulates layer 2 meanwhile): the
            // first half of each layer-1 chunk goes to slot 0, the second to slot 1
            // once layer 2 has read the chunk before it there
            drain16<kDump>(lane_addr + kColD1 + 64, bias + kB1 + 64 + 16 * q, slots + kSlot, r, q, dcol(0, 64 + 16 * q));
            publish(&B.act_h1[1]);
            for (int c = 1; c < 4; ++c) {
                wait_acc(&B.acc_d1, ph_d1);
                drain16<kDump>(lane_addr + kColD1, bias + kB1 + 128 * c + 16 * q, slots, r, q,
                               dcol(0, 128 * c + 16 * q));
                publish(&B.act_h1[0]);
                wait_acc(&B.acc_h1free, ph_free);
                drain16<kDump>(lane_addr + kColD1 + 64, bias + kB1 + 128 * c + 64 + 16 * q, slots + kSlot, r, q,
                               dcol(0, 128 * c + 64 + 16 * q));
                publish(&B.act_h1[1]);
            }
            // the next tile's row metadata: loads issued where the rows wait for
            // layer 2 anyway, consumed after layer 3
            if (has_next) issue_meta(a, next * 128 + r, nf);
            // ---- layer 2 -> h2, chunks 4,5 first (their TMEM columns become layer 3's)
            wait_acc(&B.acc_main, ph_main);
            for (int kk = 0; kk < 6; ++kk) {
                const int k = kk < 2 ? 4 + kk : kk - 2;
                drain16<kDump>(lane_addr + kColD2 + 64 * k, bias + kB2 + 64 * k + 16 * q, slots + k * kSlot, r, q,
                               dcol(1, 64 * k + 16 * q));
                publish(&B.act_h2[k]);
            }
            // ---- layer 3 -> h3 (layer 3 has read slots 4-5: stage the next tile's features there)
            wait_acc(&B.acc_main, ph_main);
            if (has_next && tid == 0) mbar_arrive(&B.feat_free);
            for (int k = 0; k < 4; ++k) {
                drain16<kDump>(lane_addr + kColD3 + 64 * k, bias + kB3 + 64 * k + 16 * q, slots + k * kSlot, r, q,
                               dcol(2, 64 * k + 16 * q));
                publish(&B.act_h3[k]);
            }
            if (has_next) nri = resolve(a, nf);                // the next tile's metadata has arrived
            // ---- layer 4 -> h4
            wait_acc(&B.acc_main, ph_main);
            for (int k = 0; k < 2; ++k) {
                drain16<kDump>(lane_addr + kColD4 + 64 * k, bias + kB4 + 64 * k + 16 * q, slots + k * kSlot, r, q,
                               dcol(3, 64 * k + 16 * q));
                publish(&B.act_h4[k]);
            }
            // ---- next tile's state row (slot 2 and TMEM [0,128) are free now): the
            // tensor pipe runs its curiosity layer 1 while the rows finish this tile's head
            if (has_next) build_x(nri);
            // ---- layer 5 + scalar head
            wait_acc(&B.acc_main, ph_main);
            {
                float v[16];
                tmem_ld16(lane_addr + kColD5, v);
                float dot = 0.f;
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const float h = bf16_round(relu(v[j] + bias[kB5 + 16 * q + j]));
                    dot = fmaf(h, bias[kHW + 16 * q + j], dot);
                    if constexpr (kDump) {
                        if (drow) drow[a.dump.crit_off[4] + 16 * q + j] = h;
                    }
                }
                part_v[q * 128 + r] = dot;
            }
            tc_fence_before();
            row_sync();
            if (q == 0) {
                const float value = ((part_v[r] + part_v[128 + r]) + (part_v[256 + r] + part_v[384 + r])) + bias[kHB];
                const float se = (part_s[r] + part_s[128 + r]) + (part_s[256 + r] + part_s[384 + r]);
                if (ri.kind == 0) {
                    a.values[ri.row] = value;
                    a.rewards[ri.row] = ri.rew + a.env.cur_coef * (se / (float)kState);
                } else if (ri.kind == 2) {
                    a.values[ri.row] = 0.f;
                } else if (ri.kind == 1) {
                    a.boot[ri.row] = value;
                } else if (ri.kind == 3) {
                    a.boot[ri.row] = 0.f;
                }
            }
            // ---- the next tile's curiosity layer 1 -> Z (slot 3 is free)
            if (has_next) cur1_epilogue(nri);
            ok = row_sync_and(ok);                             // every row warp leaves on the same tile
        }
    }
    if (abort_sh && tid == 0) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, 512);
}

}  // namespace

cudaError_t launch_value_umma(const ValueArgs &a, const UmmaWeights &w, cudaStream_t s, bool stall)
{
    if (!w.bf16 || w.wide || w.n_units != kUnits) return cudaErrorNotSupported;
    if ((reinterpret_cast<uintptr_t>(a.F) & 15u) != 0) return cudaErrorInvalidValue;   // feature copies
    for (int u = 0; u < w.n_units; ++u)
        if (w.unit_bytes[u] > (uint32_t)kStage || (w.unit_bytes[u] & 15u) || (w.unit_off[u] & 15)) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(value_umma_bf16_kernel<false, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(value_umma_bf16_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(value_umma_bf16_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmem);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long total = (long long)a.N * a.L + a.N;
    const long long tiles = (total + 127) / 128;
    const int grid = (int)(tiles < sms ? tiles : sms);
    if (stall) value_umma_bf16_kernel<true, false><<<grid, kThreads, kSmem, s>>>(a, w);
    else if (a.dump.p) value_umma_bf16_kernel<false, true><<<grid, kThreads, kSmem, s>>>(a, w);
    else value_umma_bf16_kernel<false, false><<<grid, kThreads, kSmem, s>>>(a, w);
    return cudaGetLastError();
}

}  // namespace rl
