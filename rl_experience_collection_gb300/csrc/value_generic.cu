// value_generic.cu -- tensor-core value phase for the layer shapes whose
// activations do not fit in shared memory: tf32 operands (4-byte elements) and
// the widened critic 54->1024->768->512->256->128->1.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Kernel Phases", Phase A steps 5 (critic) and 9 (curiosity, bonus =
// cur_coef * MSE against the pre-reset next state).
//
// Same roles as the bf16 kernel (16 row warps, a producer warp, an MMA warp;
// M = 128 rows per tile, f32 accumulators in TMEM), but every activation --
// the state X, the curiosity hidden Z and the critic's hidden layers -- lives
// in a per-CTA scratch region of global memory (L2-resident), written by the
// row warps as swizzled K-chunk tiles and read back by the producer with bulk
// TMA together with the matching weight tile.  Each layer runs in N-passes of
// at most 256 columns, alternating between TMEM columns [0,256) and
// [256,512) so that the rows drain one pass while the next accumulates.
//   per tile: CUR1 (A = X) -> Z; CUR2 (A = Z) -> MSE; critic 1 (A = X) -> P;
//             critic 2 (P) -> Q; critic 3 (Q) -> P; critic 4 (P) -> Q;
//             critic 5 (Q) -> scalar head.
// A layer's output buffer is the one its predecessor read, and is written only
// after that predecessor's MMAs completed (they precede it in issue order).
#include "env.cuh"
#include "umma.cuh"
#include "umma_path.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kRowWarps = 16;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kThreads = kRowThreads + 64;
constexpr int kChunk = 128 * 128;              // one 128-row K-chunk tile
constexpr int kAStage = kChunk;
constexpr int kBStage = 256 * 128;
constexpr int kStageBytes = kAStage + kBStage;
constexpr int kStages = 4;
// shared-memory copy of the epilogue constants: every job's bias (each padded
// to a multiple of 64 columns), the head weights and the curiosity one-hot
// columns (rows padded to kOhLd floats, so the rows of different actions start
// on different banks); sized for the widened critic, the larger of the two
// shapes the library accepts
constexpr int kOhLd = kCurH + 4;
constexpr int kVecCap = (1024 + 768 + 512 + 256 + 128 + 64 + 64) + 128 + kActions * kOhLd;
constexpr int kSmem = kStages * kStageBytes + 2 * 4 * 128 * 4 + kVecCap * 4 + 1024;
static_assert(kSmem <= 232448, "generic value kernel shared memory");

enum { kBufX = 0, kBufZ = 1, kBufP = 2, kBufQ = 3 };
enum { kEpiHidden = 0, kEpiHead = 1, kEpiCur1 = 2, kEpiCur2 = 3 };

struct Job {
    int layer;       // index into w.job
    int in_buf, out_buf, epi;
};
// execution order: curiosity first, then the critic
__constant__ const Job kJobs[7] = {
    {kJobCur1, kBufX, kBufZ, kEpiCur1}, {kJobCur2, kBufZ, -1, kEpiCur2},
    {kJobCrit1, kBufX, kBufP, kEpiHidden}, {kJobCrit2, kBufP, kBufQ, kEpiHidden},
    {kJobCrit3, kBufQ, kBufP, kEpiHidden}, {kJobCrit4, kBufP, kBufQ, kEpiHidden},
    {kJobCrit5, kBufQ, -1, kEpiHead},
};

struct GBars {
    uint64_t full[kStages], empty[kStages];
    uint64_t act;              // rows -> producer: a layer's input is complete (one phase per layer)
    uint64_t acc[2];           // MMA -> rows: N-pass accumulated in TMEM half h
    uint64_t tfree[2];         // rows -> MMA: TMEM half h drained
    uint64_t final_;
};

template <bool BF16>
struct Geo {
    static constexpr int EB = BF16 ? 2 : 4;
    static constexpr int KC = 128 / EB;        // elements per K-chunk
};

__device__ __forceinline__ float round_op(float x, bool bf16)
{
    return bf16 ? __uint_as_float(pack_bf16x2(0.f, x) & 0xFFFF0000u) : __uint_as_float(to_tf32(x));
}

// 16 values of row r, logical columns [c0, c0+16) (c0 a multiple of 16) into a
// buffer of swizzled K-chunk tiles
template <bool BF16>
__device__ __forceinline__ void put16g(uint8_t *buf, int r, int c0, const float (&v)[16])
{
    constexpr int KC = Geo<BF16>::KC;
    if constexpr (BF16) {
        uint8_t *tile = buf + (size_t)(c0 / KC) * kChunk;
        const int u0 = (c0 % KC) / 8;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            uint4 p;
            p.x = pack_bf16x2(v[8 * h + 0], v[8 * h + 1]);
            p.y = pack_bf16x2(v[8 * h + 2], v[8 * h + 3]);
            p.z = pack_bf16x2(v[8 * h + 4], v[8 * h + 5]);
            p.w = pack_bf16x2(v[8 * h + 6], v[8 * h + 7]);
            *reinterpret_cast<uint4 *>(tile + sw128_offset(r, u0 + h)) = p;
        }
    } else {
        uint8_t *tile = buf + (size_t)(c0 / KC) * kChunk;
        const int u0 = (c0 % KC) / 4;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            uint4 p;
            p.x = to_tf32(v[4 * h + 0]);
            p.y = to_tf32(v[4 * h + 1]);
            p.z = to_tf32(v[4 * h + 2]);
            p.w = to_tf32(v[4 * h + 3]);
            *reinterpret_cast<uint4 *>(tile + sw128_offset(r, u0 + h)) = p;
        }
    }
}

__device__ __forceinline__ void tmem_ld16g(uint32_t taddr, float (&v)[16])
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

__device__ __forceinline__ void fence_async_global()
{
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ void row_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kRowThreads) : "memory"); }

// row_sync that also returns the AND of `pred` over every row thread: a wait
// that expired in one row warp may have succeeded in another, and all row
// warps must leave the tile loop together (they share barrier 1)
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

struct RowInfoG {
    int kind;            // 0 tuple, 1 bootstrap row, 2 tuple of an invalid episode, 3 bootstrap of one, -1 none
    long long row, bar;
    int act;
    float vin, ein, vpost, epost;
};

__device__ __forceinline__ RowInfoG decode_g(const ValueArgs &a, long long r)
{
    RowInfoG ri{};
    ri.kind = -1;
    const long long NL = (long long)a.N * a.L;
    const int L = a.L;
    if (r < NL) {
        const int n = (int)(r / L), t = (int)(r % L);
        const int start = __ldg(a.starts + n);
        ri.row = r;
        if (start_ok(start, L, a.n_bars)) {
            ri.kind = 0;
            ri.bar = (long long)start + t;
            ri.act = a.actions[r];
            ri.vin = a.values[r];
            ri.vpost = a.v_post[r];
            ri.epost = exposure_of(ri.act);
            ri.ein = (t == 0 || a.dones[r - 1]) ? 0.f : exposure_of(a.actions[r - 1]);
        } else {
            ri.kind = 2;
        }
    } else if (r < NL + a.N) {
        const int n = (int)(r - NL);
        const int start = __ldg(a.starts + n);
        const long long last = (long long)n * L + L - 1;
        ri.row = last;
        if (start_ok(start, L, a.n_bars)) {
            ri.kind = 1;
            ri.bar = (long long)start + L;
            ri.act = a.actions[last];
            ri.vin = a.v_post[last];
            ri.ein = exposure_of(ri.act);
        } else {
            ri.kind = 3;
        }
    }
    return ri;
}

// one arrival per warp once every lane has passed its fences (the barriers
// count warps: per-thread arrivals on one barrier serialise in the
// shared-memory atomic unit)
__device__ __forceinline__ void warp_arrive(uint64_t *bar)
{
    __syncwarp();
    if ((threadIdx.x & 31) == 0) mbar_arrive(bar);
}

// the test hook's row of a tile row (ActDump), or nullptr
__device__ __forceinline__ float *dump_row_g(const ValueArgs &a, const RowInfoG &ri)
{
    if (ri.kind != 0 && ri.kind != 1) return nullptr;
    const long long n = ri.row / a.L;
    return a.dump.row(n, ri.kind == 0 ? (int)(ri.row - n * a.L) : a.L, a.L);
}

// the operand values v (as the next layer reads them) to dst[0..16), columns
// below n_valid only
template <bool BF16>
__device__ __forceinline__ void dump16(float *dst, const float (&v)[16], int c0, int n_valid)
{
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (c0 + i < n_valid) dst[i] = round_op(v[i], BF16);
}

// kStall: a test build in which the producer of CTA 0 issues no copy, so that
// CTA's MMA issuer waits on a stage that never fills and the bounded-wait exit
// runs (rollout_test_stall).  kDump: a test build that also writes every
// row's rounded hidden activations (rollout_test_activations).
template <bool BF16, bool kStall, bool kDump>
__global__ void __launch_bounds__(kThreads, 1) value_generic_kernel(ValueArgs a, UmmaWeights w, uint8_t *scratch,
                                                                    long long scratch_per_cta)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    uint8_t *ring = sm;
    float *part = reinterpret_cast<float *>(ring + kStages * kStageBytes);   // [2][4][128]
    float *vc = part + 2 * 4 * 128;                                            // [kVecCap] epilogue constants
    __shared__ __align__(8) GBars B;
    __shared__ uint32_t tmem_base_sh;
    __shared__ int abort_sh;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // scratch buffers of this CTA: X and Z (2 chunks each), P and Q (widest layer)
    uint8_t *my = scratch + (long long)blockIdx.x * scratch_per_cta;
    const long long big = (scratch_per_cta - 4LL * kChunk) / 2;
    uint8_t *bufs[4] = {my, my + 2 * kChunk, my + 4 * kChunk, my + 4 * kChunk + big};

    if (tid == 0) {
        abort_sh = 0;
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&B.full[s], 1);
            mbar_init(&B.empty[s], 1);
        }
        mbar_init(&B.act, kRowWarps);
        for (int h = 0; h < 2; ++h) {
            mbar_init(&B.acc[h], 1);
            mbar_init(&B.tfree[h], kRowWarps);
        }
        mbar_init(&B.final_, 1);
        fence_mbar_init();
    }
    if (warp == kRowWarps + 1) {
        tmem_alloc(&tmem_base_sh, 512);
        tmem_relinquish();
    }
    // epilogue constants into shared memory (offsets: jobs in execution order,
    // then the head weights, then the one-hot rows)
    int vc_n = 0;
    for (int jj = 0; jj < 7; ++jj) {
        const UmmaLayer &Ly = w.job[kJobs[jj].layer];
        const int n = (Ly.n_out + 63) & ~63;
        for (int i = tid; i < n; i += kThreads) vc[vc_n + i] = i < Ly.n_out ? w.vec[Ly.bias_off + i] : 0.f;
        vc_n += n;
    }
    const int vc_head = vc_n, vc_oh = vc_head + w.job[kJobCrit5].n_out;
    for (int i = tid; i < w.job[kJobCrit5].n_out; i += kThreads) vc[vc_head + i] = w.vec[w.head_w_off + i];
    for (int i = tid; i < kActions * kCurH; i += kThreads)
        vc[vc_oh + (i / kCurH) * kOhLd + i % kCurH] = w.vec[w.onehot_off + i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_sh;
    volatile int *abort = &abort_sh;
    const long long total = (long long)a.N * a.L + a.N;
    const long long n_tiles = (total + 127) / 128;

    if (warp == kRowWarps) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, act_ph = 0;
            bool ok = true;
            const bool silent = kStall && blockIdx.x == 0;
            for (long long tile = blockIdx.x; tile < n_tiles && ok && !silent; tile += gridDim.x) {
                for (int jj = 0; jj < 7 && ok; ++jj) {
                    const Job J = kJobs[jj];
                    const UmmaLayer &Ly = w.job[J.layer];
                    // the rows publish every layer's input (X, then each output)
                    if (J.layer != kJobCrit1) {        // critic 1 reads X, already published for CUR1
                        ok = mbar_wait(&B.act, act_ph, abort);
                        act_ph ^= 1u;
                        if (!ok) break;
                    }
                    const uint8_t *in = bufs[J.in_buf];
                    int row0 = 0;
                    for (int nb = 0; nb < Ly.n_blocks && ok; ++nb) {
                        const int rows = Ly.nb_rows[nb];
                        for (int c = 0; c < Ly.k_chunks && ok; ++c) {
                            ok = mbar_wait(&B.empty[stage], phase ^ 1u, abort);
                            if (!ok) break;
                            const uint32_t bbytes = (uint32_t)rows * 128u;
                            mbar_arrive_expect_tx(&B.full[stage], kAStage + bbytes);
                            uint8_t *st = ring + stage * kStageBytes;
                            bulk_g2s(st, in + (size_t)c * kChunk, kAStage, &B.full[stage]);
                            // weight stream: N-block-major, K-chunk tiles of the block contiguous
                            const long long off = Ly.w_off + (long long)row0 * 128 * Ly.k_chunks + (long long)c * bbytes;
                            bulk_g2s(st + kAStage, w.stream + off, bbytes, &B.full[stage]);
                            if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        }
                        row0 += rows;
                    }
                }
            }
            for (int s = 0; s < kStages && ok; ++s) {
                ok = mbar_wait(&B.empty[stage], phase ^ 1u, abort);
                if (++stage == kStages) { stage = 0; phase ^= 1u; }
            }
            if (!ok) {
                const long long c0 = clock64();
                while (clock64() - c0 < 4000000) { }
            }
        }
        __syncwarp();
    } else if (warp == kRowWarps + 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0, tf_ph[2] = {0, 0};
            int pass = 0;                               // global N-pass counter: TMEM half = pass & 1
            bool ok = true;
            const uint32_t s_ring = smem_u32(ring);
            for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
                for (int jj = 0; jj < 7 && ok; ++jj) {
                    const Job J = kJobs[jj];
                    const UmmaLayer &Ly = w.job[J.layer];
                    for (int nb = 0; nb < Ly.n_blocks && ok; ++nb, ++pass) {
                        const int h = pass & 1, rows = Ly.nb_rows[nb];
                        if (pass >= 2) {                 // the rows drained this TMEM half
                            ok = mbar_wait(&B.tfree[h], tf_ph[h], abort);
                            tf_ph[h] ^= 1u;
                            tc_fence_after();
                        }
                        const uint32_t id = idesc(BF16, 128, rows);
                        for (int c = 0; c < Ly.k_chunks && ok; ++c) {
                            ok = mbar_wait(&B.full[stage], phase, abort);
                            if (!ok) break;
                            tc_fence_after();
                            const uint32_t a0 = s_ring + stage * kStageBytes, b0 = a0 + kAStage;
#pragma unroll
                            for (int k = 0; k < 4; ++k)
                                mma<BF16>(tmem + 256 * h, desc_sw128(a0 + 32 * k), desc_sw128(b0 + 32 * k), id,
                                          (c | k) != 0);
                            mma_commit(&B.empty[stage]);
                            if (++stage == kStages) { stage = 0; phase ^= 1u; }
                        }
                        mma_commit(&B.acc[h]);
                    }
                }
            }
            mma_commit(&B.final_);
            int never = 0;
            mbar_wait(&B.final_, 0, &never, 100000000ull);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ row warps
        const int r = 32 * (warp & 3) + lane;
        const int q = warp >> 2;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * (warp & 3)) << 16);
        uint32_t acc_ph[2] = {0, 0};
        int pass = 0;
        bool ok = true;
        float *part_v = part, *part_s = part + 4 * 128;
        const float *vec = w.vec;
        for (long long tile = blockIdx.x; tile < n_tiles && ok; tile += gridDim.x) {
            const RowInfoG ri = decode_g(a, tile * 128 + r);
            const bool has = ri.kind == 0 || ri.kind == 1;
            float *drow = nullptr;                              // test hook: this row's activation dump
            if constexpr (kDump) drow = dump_row_g(a, ri);
            // ---- state row: X buffer (operand)
            {
                float xv[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const int c = 16 * q + j;
                    float x = 0.f;
                    if (has) {
                        if (c < kMarket) x = __ldg(a.F + ri.bar * kMarket + c);
                        else if (c == kMarket) x = ri.vin;
                        else if (c == kMarket + 1) x = ri.ein;
                        else if (c == kMarket + 2) x = a.env.spread;
                    }
                    xv[j] = x;
                }
                put16g<BF16>(bufs[kBufX], r, 16 * q, xv);
                if constexpr (kDump) {
                    if (drow) dump16<BF16>(drow + 16 * q, xv, 16 * q, kState);
                }
            }
            fence_async_global();
            warp_arrive(&B.act);
            float se = 0.f, dot = 0.f;
            int vc_off = 0;                           // this job's bias in vc (64-column padded)
            for (int jj = 0; jj < 7; ++jj) {
                const Job J = kJobs[jj];
                const UmmaLayer &Ly = w.job[J.layer];
                const float *bias = vc + vc_off;
                vc_off += (Ly.n_out + 63) & ~63;
                int col0 = 0;
                for (int nb = 0; nb < Ly.n_blocks; ++nb, ++pass) {
                    const int h = pass & 1, rows = Ly.nb_rows[nb];
                    ok = __all_sync(0xffffffffu, ok && mbar_wait(&B.acc[h], acc_ph[h], abort));
                    acc_ph[h] ^= 1u;
                    tc_fence_after();
                    // this thread drains columns [64g + 16q, +16) of every 64-column group
                    for (int g = 0; g < rows / 64; ++g) {
                        const int cl = 64 * g + 16 * q;          // column within the pass
                        const int cg = col0 + cl;                // column within the layer
                        float v[16];
                        tmem_ld16g(lane_addr + 256 * h + cl, v);
                        float bv[16];
                        {
                            const float4 *b4 = reinterpret_cast<const float4 *>(bias + cg);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float4 b = b4[k];
                                bv[4 * k + 0] = b.x;
                                bv[4 * k + 1] = b.y;
                                bv[4 * k + 2] = b.z;
                                bv[4 * k + 3] = b.w;
                            }
                        }
                        if (J.epi == kEpiHidden) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = relu(v[i] + bv[i]);
                            put16g<BF16>(bufs[J.out_buf], r, cg, v);
                            if constexpr (kDump) {
                                if (drow) dump16<BF16>(drow + a.dump.crit_off[J.layer - kJobCrit1] + cg, v, cg, Ly.n_out);
                            }
                        } else if (J.epi == kEpiCur1) {
                            const int act = (ri.act >= 0 && ri.act < kActions) ? ri.act : 0;
                            const float4 *oh4 = reinterpret_cast<const float4 *>(vc + vc_oh + act * kOhLd + cg);
#pragma unroll
                            for (int k = 0; k < 4; ++k) {
                                const float4 o = oh4[k];
                                v[4 * k + 0] = relu((v[4 * k + 0] + o.x) + bv[4 * k + 0]);
                                v[4 * k + 1] = relu((v[4 * k + 1] + o.y) + bv[4 * k + 1]);
                                v[4 * k + 2] = relu((v[4 * k + 2] + o.z) + bv[4 * k + 2]);
                                v[4 * k + 3] = relu((v[4 * k + 3] + o.w) + bv[4 * k + 3]);
                            }
                            put16g<BF16>(bufs[J.out_buf], r, cg, v);
                            if constexpr (kDump) {
                                if (drow && ri.kind == 0) dump16<BF16>(drow + a.dump.cur_off + cg, v, cg, Ly.n_out);
                            }
                        } else if (J.epi == kEpiCur2) {
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int c = cg + i;
                                if (c < kState) {
                                    float tgt = a.env.spread;
                                    if (c < kMarket) tgt = ri.kind == 0 ? __ldg(a.F + (ri.bar + 1) * kMarket + c) : 0.f;
                                    else if (c == kMarket) tgt = ri.vpost;
                                    else if (c == kMarket + 1) tgt = ri.epost;
                                    const float d = (v[i] + bv[i]) - tgt;
                                    se = fmaf(d, d, se);
                                }
                            }
                        } else {   // head: relu, operand rounding, dot with the head weights
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const float hv = round_op(relu(v[i] + bv[i]), BF16);
                                dot = fmaf(hv, vc[vc_head + cg + i], dot);
                                if constexpr (kDump) {
                                    if (drow && cg + i < Ly.n_out) drow[a.dump.crit_off[4] + cg + i] = hv;
                                }
                            }
                        }
                    }
                    col0 += rows;
                    // TMEM half drained (and, for the last pass of a layer, its output written)
                    fence_async_global();
                    tc_fence_before();
                    warp_arrive(&B.tfree[h]);
                }
                if (J.out_buf >= 0) warp_arrive(&B.act);     // this layer's output is complete
            }
            part_v[q * 128 + r] = dot;
            part_s[q * 128 + r] = se;
            row_sync();
            if (q == 0) {
                const float value = ((part_v[r] + part_v[128 + r]) + (part_v[256 + r] + part_v[384 + r])) +
                                    __ldg(vec + w.head_b_off);
                const float s2 = (part_s[r] + part_s[128 + r]) + (part_s[256 + r] + part_s[384 + r]);
                if (ri.kind == 0) {
                    a.values[ri.row] = value;
                    a.rewards[ri.row] += a.env.cur_coef * (s2 / (float)kState);
                } else if (ri.kind == 2) {
                    a.values[ri.row] = 0.f;
                } else if (ri.kind == 1) {
                    a.boot[ri.row] = value;
                } else if (ri.kind == 3) {
                    a.boot[ri.row] = 0.f;
                }
            }
            ok = row_sync_and(ok);                             // every row warp leaves on the same tile
        }
    }
    if (abort_sh && tid == 0) set_status(a.status, ROLLOUT_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kRowWarps + 1) tmem_dealloc(tmem, 512);
}

template <bool BF16>
cudaError_t launch_g(const ValueArgs &a, const UmmaWeights &w, uint8_t *scratch, long long per_cta, int grid,
                     cudaStream_t s, bool stall)
{
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(value_generic_kernel<BF16, false, false>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(value_generic_kernel<BF16, true, false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(value_generic_kernel<BF16, false, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    if (stall) value_generic_kernel<BF16, true, false><<<grid, kThreads, kSmem, s>>>(a, w, scratch, per_cta);
    else if (a.dump.p) value_generic_kernel<BF16, false, true><<<grid, kThreads, kSmem, s>>>(a, w, scratch, per_cta);
    else value_generic_kernel<BF16, false, false><<<grid, kThreads, kSmem, s>>>(a, w, scratch, per_cta);
    return cudaGetLastError();
}

}  // namespace

long long value_generic_scratch_per_cta(const UmmaWeights &w)
{
    // X and Z: two K-chunk tiles each; P and Q: the widest hidden layer
    int widest = 0;
    for (int j = kJobCrit1; j <= kJobCrit5; ++j) widest = w.job[j].n_out > widest ? w.job[j].n_out : widest;
    const int kc = w.bf16 ? 64 : 32;
    const long long big = (long long)((widest + kc - 1) / kc) * kChunk;
    return 4LL * kChunk + 2 * big;
}

cudaError_t launch_value_generic(const ValueArgs &a, const UmmaWeights &w, uint8_t *scratch, long long per_cta,
                                 int grid, cudaStream_t s, bool stall)
{
    for (int j = 0; j < kNumJobs; ++j) {
        const UmmaLayer &L = w.job[j];
        int rows = 0;
        for (int nb = 0; nb < L.n_blocks; ++nb) {
            if (L.nb_rows[nb] > 256 || L.nb_rows[nb] % 64) return cudaErrorInvalidValue;
            rows += L.nb_rows[nb];
        }
        if (L.k_chunks > 16) return cudaErrorInvalidValue;
    }
    return w.bf16 ? launch_g<true>(a, w, scratch, per_cta, grid, s, stall)
                  : launch_g<false>(a, w, scratch, per_cta, grid, s, stall);
}

}  // namespace rl
