// ppo_gemm.cu -- the dense products of the on-device PPO update on the tensor
// cores: C[M, N] = A[M, K] B[N, K]^T with float32 operands and results.
//
// Page "Fused CUDA Training Kernel -- Implementation Plan", "Chunk 2:
// Backward Pass Kernel" (the linear layers' weight gradient dW = dY^T X, bias
// gradient db = sum of dY over the rows, and input gradient dX = dY W, masked
// by the activation's derivative); the forward products are the MLP layers of
// page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// section "Weight Layout" ([out, in] row-major weights).
//
// Precision: every float32 operand x is split into two bf16 values, hi =
// bf16(x) and lo = bf16(x - hi), so that |x - hi - lo| <= 2^-18 |x|, and each
// product is taken as hi*hi + hi*lo + lo*hi (three tcgen05 kind::f16 MMAs,
// float32 accumulation in tensor memory).  The dropped lo*lo term and the
// split's remainder keep each product within about 1.2e-5 of the float32
// product, far inside the update's parity tolerances, so the float32 oracle
// stays the reference.
//
// One CTA (16 warps) computes a 128 x 128 tile of C: its threads load the
// tile's K-chunks of A and B (64 elements each, zero outside the matrices),
// split them into swizzled bf16 operand tiles in shared memory (two stages, so
// that loading chunk c + 1 overlaps the MMAs of chunk c), one thread issues
// the MMAs, and after the last chunk the accumulator goes from tensor memory
// (each warp reads its lane quadrant's share of the columns) through shared
// memory, so that every global write is coalesced, into the epilogue:
//   forward:         Y = C + bias (ReLU for hidden layers), and Y^T
//   weight gradient: C[:, :nw] into dW, column nw into db (the B operand's
//                    row nw is all ones: the column sums of dY)
//   input gradient:  Y = C where H > 0, else 0 (ReLU'), and Y^T
// Where float32 products are needed to float32 rounding (a forward pass of
// float32 networks), each operand is split three ways, hi + mid + lo, and the
// six products of parts above 2^-23 relative are taken.
// For a forward pass in the collector's own operand format the operands are
// instead rounded once to bf16 (one kind::f16 MMA per K-step) or to tf32 (one
// kind::tf32 MMA per K-step over two 32-element tiles).
// A product whose K spans many chunks is split along K: each of its ksplit
// CTAs per tile writes its partial tile to a workspace, and the CTA that
// arrives last at the tile's counter (atomic ticket, reset by that CTA) adds
// the partials in split order and runs the epilogue, so the sum's order is
// fixed.  Several independent products share one launch (blockIdx.x runs over
// the tiles and splits of all of them).
// Every wait is bounded; a CTA that gives up sets ROLLOUT_ERR_TIMEOUT.
#include "env.cuh"
#include "pdl.cuh"
#include "ppo_gemm.cuh"
#include "umma.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kBM = kGemmTile, kBN = kGemmTile, kBK = kGemmChunk;   // tile rows, columns, K elements per chunk
constexpr int kTile = 128 * 128;                           // bytes of one 128-row bf16 operand tile
constexpr int kStageBytes = 6 * kTile;                     // A hi, A lo, B hi, B lo (, A mid, B mid)
constexpr int kGemmSmem = 2 * kStageBytes + 1024;          // two stages + alignment slack
constexpr int kWarps = 16;
constexpr int kGemmThreads = 32 * kWarps;
constexpr int kRuns = (kBM * kBK / 4) / kGemmThreads;      // runs of four elements per thread and operand
constexpr int kMaxSplitG = 4;                              // most K-splits of one product
constexpr int kLd = kBN + 1;                               // row stride of the staged tile (floats)

// the bf16 pair (hi, lo) of x
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo)
{
    const uint32_t h = pack_bf16x2(0.f, x) & 0xFFFF0000u;   // nearest-even bf16 of x (upper half)
    hi = __uint_as_float(h);
    lo = x - hi;                                             // exact in float32
}

// K-chunk c of rows [r0, r0 + 128) of X [rows, K] (row stride ld), held in
// registers: thread t takes kRuns runs of four elements (zero outside X), as
// one 16-byte load where the run is whole and aligned (vec: ld a multiple of
// 4 and X 16-byte aligned).  All loads are issued before any is used, so a
// chunk costs one round trip to L2.
struct Runs {
    float v[kRuns][4];
};

__device__ __forceinline__ void load_runs(const float *X, int ld, int rows, int K, int r0, int c, bool vec, Runs &R)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int s = 0; s < kRuns; ++s) {
        const int j = tid + kGemmThreads * s;                   // run of four elements
        const int r = j >> 4, q = j & 15;                        // row, run within the row
        const int row = r0 + r, col = c * kBK + 4 * q;
        const float *src = X + (long long)row * ld + col;
        if (vec && row < rows && col + 3 < K) {
            const float4 f = __ldg(reinterpret_cast<const float4 *>(src));
            R.v[s][0] = f.x;
            R.v[s][1] = f.y;
            R.v[s][2] = f.z;
            R.v[s][3] = f.w;
        } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) R.v[s][i] = (row < rows && col + i < K) ? __ldg(src + i) : 0.f;
        }
    }
}

// the runs split into the swizzled hi / lo operand tiles
__device__ __forceinline__ void store_split(const Runs &R, uint8_t *hi_tile, uint8_t *lo_tile)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int s = 0; s < kRuns; ++s) {
        const int j = tid + kGemmThreads * s;
        const int r = j >> 4, q = j & 15;
        float h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_bf16(R.v[s][i], h[i], l[i]);
        const uint2 ph = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
        const uint2 pl = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
        const uint32_t off = sw128_offset(r, q >> 1) + 8 * (q & 1);   // 16-byte unit q/2 of row r, half q%2
        *reinterpret_cast<uint2 *>(hi_tile + off) = ph;
        *reinterpret_cast<uint2 *>(lo_tile + off) = pl;
    }
}

// the runs rounded to one operand format into two swizzled tiles: bf16
// (K elements 0..63 of the chunk in `t0`; `t1` unused) or tf32 (elements 0..31
// in `t0`, 32..63 in `t1`, four bytes each)
template <int OPS>
__device__ __forceinline__ void store_round(const Runs &R, uint8_t *t0, uint8_t *t1)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int s = 0; s < kRuns; ++s) {
        const int j = tid + kGemmThreads * s;
        const int r = j >> 4, q = j & 15;
        if constexpr (OPS == kGemmBf16) {
            const uint2 p = make_uint2(pack_bf16x2(R.v[s][0], R.v[s][1]), pack_bf16x2(R.v[s][2], R.v[s][3]));
            *reinterpret_cast<uint2 *>(t0 + sw128_offset(r, q >> 1) + 8 * (q & 1)) = p;
        } else {
            const uint4 p = make_uint4(to_tf32(R.v[s][0]), to_tf32(R.v[s][1]), to_tf32(R.v[s][2]), to_tf32(R.v[s][3]));
            *reinterpret_cast<uint4 *>((q < 8 ? t0 : t1) + sw128_offset(r, q & 7)) = p;
        }
    }
}

// the runs split three ways (x = hi + mid + lo, |x - hi - mid - lo| <= 2^-27 |x|)
// into the swizzled hi / mid / lo tiles
__device__ __forceinline__ void store_split3(const Runs &R, uint8_t *hi_tile, uint8_t *mid_tile, uint8_t *lo_tile)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int s = 0; s < kRuns; ++s) {
        const int j = tid + kGemmThreads * s;
        const int r = j >> 4, q = j & 15;
        float h[4], m[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float r1;
            split_bf16(R.v[s][i], h[i], r1);
            split_bf16(r1, m[i], l[i]);
        }
        const uint32_t off = sw128_offset(r, q >> 1) + 8 * (q & 1);
        *reinterpret_cast<uint2 *>(hi_tile + off) = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
        *reinterpret_cast<uint2 *>(mid_tile + off) = make_uint2(pack_bf16x2(m[0], m[1]), pack_bf16x2(m[2], m[3]));
        *reinterpret_cast<uint2 *>(lo_tile + off) = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
    }
}

struct GemmGroup {
    GemmArgs g[kGemmGroup];
    int n;
    int first[kGemmGroup + 1];   // first block of each product
};

// The epilogue of the staged tile (rows [0, nrows), columns [0, ncols) of
// `stage`), one instantiation per kind of product.  Warp w takes rows w,
// w + 16, ... (eight at a time); lane l columns l, l + 32, ... of each
// (consecutive lanes: consecutive addresses); bounds are predicates on the
// accesses.
// The same with 16-byte accesses: lane l takes columns 4 l .. 4 l + 3 of a
// row (a warp one whole 128-column row per instruction), and in the transposed
// pass rows 4 l .. 4 l + 3 of a column.  Used when the row strides and base
// addresses allow it and the tile is whole in the directions it stores.
template <int EPI>
__device__ __forceinline__ void epilogue_vec(const GemmArgs &g, float *stage, int m0, int n0, int nrows, int ncols)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cc = 4 * lane, n = n0 + cc;
    const bool cin = cc < ncols;                             // ncols is a multiple of 4
    float4 bj = make_float4(0.f, 0.f, 0.f, 0.f);
    if (EPI == kGemmFwd && cin) bj = __ldg(reinterpret_cast<const float4 *>(g.bias + n));
    for (int rr = warp; rr < nrows; rr += kWarps) {
        const long long m = m0 + rr;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = cin ? stage[rr * kLd + cc + i] : 0.f;
        if (EPI == kGemmFwd) {
            v[0] += bj.x;
            v[1] += bj.y;
            v[2] += bj.z;
            v[3] += bj.w;
            if (g.relu) {
#pragma unroll
                for (int i = 0; i < 4; ++i) v[i] = relu(v[i]);
            }
        }
        if (EPI == kGemmDx && cin) {
            const float4 h = __ldg(reinterpret_cast<const float4 *>(g.H + m * g.ldh + n));
            v[0] = h.x > 0.f ? v[0] : 0.f;
            v[1] = h.y > 0.f ? v[1] : 0.f;
            v[2] = h.z > 0.f ? v[2] : 0.f;
            v[3] = h.w > 0.f ? v[3] : 0.f;
        }
        if (cin) {
            *reinterpret_cast<float4 *>(g.Y + m * g.ldy + n) = make_float4(v[0], v[1], v[2], v[3]);
#pragma unroll
            for (int i = 0; i < 4; ++i) stage[rr * kLd + cc + i] = v[i];   // for the transposed pass
        }
    }
    if (g.YT) {
        __syncthreads();
        const int r4 = 4 * lane;                             // nrows is a multiple of 4
        for (int c0 = warp; c0 < ncols; c0 += kWarps) {
            if (r4 < nrows) {
                float *dst = g.YT + (long long)(n0 + c0) * g.ldt + m0 + r4;
                *reinterpret_cast<float4 *>(dst) = make_float4(stage[r4 * kLd + c0], stage[(r4 + 1) * kLd + c0],
                                                               stage[(r4 + 2) * kLd + c0], stage[(r4 + 3) * kLd + c0]);
            }
        }
    }
}

template <int EPI>
__device__ __forceinline__ void epilogue(const GemmArgs &g, float *stage, int m0, int n0, int nrows, int ncols)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int jb = (ncols + 31) >> 5;                        // column blocks in use (CTA-uniform)
    for (int j = 0; j < jb; ++j) {
        const int cc = lane + 32 * j;
        const bool cin = cc < ncols;
        const int n = n0 + cc;
        float bj = 0.f;
        if (EPI == kGemmFwd) bj = cin ? __ldg(g.bias + n) : 0.f;
        for (int r0 = warp; r0 < nrows; r0 += 8 * kWarps) {
            float y[8], h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = r0 + kWarps * i;
                const bool in = cin && rr < nrows;
                y[i] = in ? stage[rr * kLd + cc] : 0.f;
                h[i] = 1.f;
                if (EPI == kGemmDx) h[i] = in ? __ldg(g.H + (long long)(m0 + rr) * g.ldh + n) : 0.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int rr = r0 + kWarps * i;
                const bool in = cin && rr < nrows;
                float v = y[i];
                if (EPI == kGemmFwd) {
                    v += bj;
                    if (g.relu) v = relu(v);
                }
                if (EPI == kGemmDx) v = h[i] > 0.f ? v : 0.f;
                const long long m = m0 + rr;
                if (EPI == kGemmDw) {
                    if (in && n < g.nw) g.Y[m * g.ldy + n] = v;
                    if (in && n == g.nw) g.db[m] = v;
                } else if (in) {
                    g.Y[m * g.ldy + n] = v;
                    stage[rr * kLd + cc] = v;                      // for the transposed pass
                }
            }
        }
    }
    if (EPI != kGemmDw && g.YT) {
        __syncthreads();
        // transposed pass: warp w takes columns w, w + 16, ..., lane l rows l, l + 32, ...
        for (int c0 = warp; c0 < ncols; c0 += kWarps) {
            float *dst = g.YT + (long long)(n0 + c0) * g.ldt + m0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int rr = lane + 32 * j;
                if (rr < nrows) dst[rr] = stage[rr * kLd + c0];
            }
        }
    }
}

// one CTA of product g (block `local` of its blocks); g is a member of the
// kernel's parameter block selected with a constant index, so that its fields
// are parameter-space reads that no global store can alias
__device__ __forceinline__ void gemm_cta(const GemmArgs &g, int local, uint8_t *sm)
{
    __shared__ __align__(8) uint64_t bar_done[2], bar_final;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    __shared__ unsigned int ticket_sh;
    // the staged accumulator, named through the dynamic shared-memory array so
    // that the compiler knows it cannot alias the global outputs
    extern __shared__ uint8_t smem_raw[];
    float *stage = reinterpret_cast<float *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // the tile and split this block computes
    const int z = local % g.ksplit, tile = local / g.ksplit;
    const int mt = (g.M + kBM - 1) / kBM;
    const int m0 = (tile % mt) * kBM, n0 = (tile / mt) * kBN;
    const int chunks = (g.K + kBK - 1) / kBK;
    const int c_begin = g.ksplit > 1 ? z * g.chunks_per_split : 0;
    const int c_end = g.ksplit > 1 ? min(chunks, c_begin + g.chunks_per_split) : chunks;
    const bool vec_a = (g.lda & 3) == 0 && ((uintptr_t)g.A & 15) == 0;
    const bool vec_b = (g.ldb & 3) == 0 && ((uintptr_t)g.B & 15) == 0;
    if (tid == 0) {
        abort_sh = 0;
        mbar_init(&bar_done[0], 1);
        mbar_init(&bar_done[1], 1);
        mbar_init(&bar_final, 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(&tmem_sh, kBN);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    // the set-up above overlaps the kernel ahead on the stream; its outputs are
    // read from here on
    pdl_wait();
    const uint32_t tmem = tmem_sh;
    volatile int *abort = &abort_sh;
    constexpr uint32_t id = idesc(true, kBM, kBN);
    bool ok = true;
    // software pipeline: the loads of chunk c + 1 are in flight while chunk c
    // is split into its stage and its MMAs are issued
    Runs ra, rb;
    if (c_begin < c_end) {
        load_runs(g.A, g.lda, g.M, g.K, m0, c_begin, vec_a, ra);
        load_runs(g.B, g.ldb, g.N, g.K, n0, c_begin, vec_b, rb);
    }
    for (int c = c_begin; c < c_end; ++c) {
        const int i = c - c_begin, s = i & 1;
        uint8_t *st = sm + s * kStageBytes;
        // the MMAs of chunk i - 2 read this stage: wait until they are done
        if (i >= 2) ok = __syncthreads_and(ok && mbar_wait(&bar_done[s], (uint32_t)(((i - 2) >> 1) & 1), abort));
        if (!ok) break;
        if (g.operands == kGemmSplit) {
            store_split(ra, st, st + kTile);
            store_split(rb, st + 2 * kTile, st + 3 * kTile);
        } else if (g.operands == kGemmSplit3) {
            store_split3(ra, st, st + 4 * kTile, st + kTile);
            store_split3(rb, st + 2 * kTile, st + 5 * kTile, st + 3 * kTile);
        } else if (g.operands == kGemmBf16) {
            store_round<kGemmBf16>(ra, st, st + kTile);
            store_round<kGemmBf16>(rb, st + 2 * kTile, st + 3 * kTile);
        } else {
            store_round<kGemmTf32>(ra, st, st + kTile);
            store_round<kGemmTf32>(rb, st + 2 * kTile, st + 3 * kTile);
        }
        if (c + 1 < c_end) {
            load_runs(g.A, g.lda, g.M, g.K, m0, c + 1, vec_a, ra);
            load_runs(g.B, g.ldb, g.N, g.K, n0, c + 1, vec_b, rb);
        }
        fence_async_smem();                       // generic-proxy stores -> visible to the tensor core
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a_hi = smem_u32(st), a_lo = a_hi + kTile, b_hi = a_hi + 2 * kTile, b_lo = a_hi + 3 * kTile;
            if (g.operands == kGemmSplit) {
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
                    mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_hi + 32 * k), id, acc);
                    mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_lo + 32 * k), id, 1u);
                    mma<true>(tmem, desc_sw128(a_lo + 32 * k), desc_sw128(b_hi + 32 * k), id, 1u);
                }
            } else if (g.operands == kGemmSplit3) {
                const uint32_t a_mi = a_hi + 4 * kTile, b_mi = a_hi + 5 * kTile;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const uint32_t acc = (i > 0 || k > 0) ? 1u : 0u;
                    // every product of parts down to 2^-16 relative: the dropped ones are below 2^-23
                    mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_hi + 32 * k), id, acc);
                    mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_mi + 32 * k), id, 1u);
                    mma<true>(tmem, desc_sw128(a_mi + 32 * k), desc_sw128(b_hi + 32 * k), id, 1u);
                    mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_lo + 32 * k), id, 1u);
                    mma<true>(tmem, desc_sw128(a_lo + 32 * k), desc_sw128(b_hi + 32 * k), id, 1u);
                    mma<true>(tmem, desc_sw128(a_mi + 32 * k), desc_sw128(b_mi + 32 * k), id, 1u);
                }
            } else if (g.operands == kGemmBf16) {
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_hi + 32 * k), id, (i > 0 || k > 0) ? 1u : 0u);
            } else {
                constexpr uint32_t idt = idesc(false, kBM, kBN);
#pragma unroll
                for (int t = 0; t < 2; ++t)
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        mma<false>(tmem, desc_sw128((t ? a_lo : a_hi) + 32 * k), desc_sw128((t ? b_lo : b_hi) + 32 * k),
                                   idt, (i > 0 || t > 0 || k > 0) ? 1u : 0u);
            }
            mma_commit(&bar_done[s]);
        }
    }
    // every MMA issued has completed before the accumulator is read (and TMEM released)
    if (tid == 0) mma_commit(&bar_final);
    {
        int never = 0;
        const bool fin = mbar_wait(&bar_final, 0, &never, 2000000000ull);
        ok = __syncthreads_and(ok && fin);
    }
    tc_fence_after();
    // tensor memory -> stage[r][c] (the operand stages are free now): warp w
    // reads lane quadrant w % 4, columns [32 (w / 4), +32); row stride kLd so
    // that rows and columns are both read without bank conflicts
    const int ncols = min(kBN, g.N - n0), nrows = min(kBM, g.M - m0);
    const bool has = c_end > c_begin;            // a split past the last chunk holds zeros
    if (ok) {
        const int q = warp & 3, cb = 32 * (warp >> 2);
        const int r = 32 * q + lane;
        float v[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + cb, v);
        tmem_ld_wait();
        if (cb < ncols) {
#pragma unroll
            for (int j = 0; j < 32; ++j) stage[r * kLd + cb + j] = has ? v[j] : 0.f;
        }
    }
    __syncthreads();
    bool fin_here = ok && g.ksplit == 1;          // this CTA runs the epilogue
    if (ok && g.ksplit > 1) {
        // this split's partial tile (warp w: rows w, w + 16, ...; coalesced), then
        // the tile's arrival ticket
        float *part = g.ws + ((long long)tile * g.ksplit + z) * (kBM * kBN);
        const int jb = (ncols + 31) >> 5;
        for (int rr = warp; rr < kBM; rr += kWarps)
            for (int j = 0; j < jb; ++j) {
                const int cc = lane + 32 * j;
                if (cc < ncols) part[rr * kBN + cc] = stage[rr * kLd + cc];
            }
        __threadfence();
        __syncthreads();
        if (tid == 0) ticket_sh = atomicAdd(g.cnt + tile, 1u);
        __syncthreads();
        if (ticket_sh == (unsigned int)(g.ksplit - 1)) {
            // the last split of this tile: the partials added in split order
            __threadfence();
            const float *base = g.ws + (long long)tile * g.ksplit * (kBM * kBN);
            for (int j = 0; j < jb; ++j) {
                const int cc = lane + 32 * j;
                for (int r0 = warp; r0 < nrows; r0 += 8 * kWarps) {
                    float acc[8], p[kMaxSplitG - 1][8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const int rr = r0 + kWarps * i;
                        const bool in = cc < ncols && rr < nrows;
                        acc[i] = in ? __ldcg(base + rr * kBN + cc) : 0.f;
#pragma unroll
                        for (int zz = 1; zz < kMaxSplitG; ++zz)
                            p[zz - 1][i] = (in && zz < g.ksplit)
                                               ? __ldcg(base + (long long)zz * (kBM * kBN) + rr * kBN + cc)
                                               : 0.f;
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
#pragma unroll
                        for (int zz = 1; zz < kMaxSplitG; ++zz)
                            if (zz < g.ksplit) acc[i] += p[zz - 1][i];
                        const int rr = r0 + kWarps * i;
                        if (cc < ncols && rr < nrows) stage[rr * kLd + cc] = acc[i];
                    }
                }
            }
            if (tid == 0) g.cnt[tile] = 0u;                        // ready for the next launch
            __syncthreads();
            fin_here = true;
        }
    }
    if (fin_here) {
        // 16-byte accesses where every row start is 16-byte aligned and the tile's
        // extents are multiples of 4 (the weight-gradient product keeps the
        // scalar form: its last column is the bias gradient)
        const bool vec = g.epi != kGemmDw && (ncols & 3) == 0 && (nrows & 3) == 0 && (g.ldy & 3) == 0 &&
                         ((uintptr_t)g.Y & 15) == 0 &&
                         (g.epi != kGemmFwd || ((uintptr_t)g.bias & 15) == 0) &&
                         (g.epi != kGemmDx || ((g.ldh & 3) == 0 && ((uintptr_t)g.H & 15) == 0)) &&
                         (!g.YT || ((g.ldt & 3) == 0 && ((uintptr_t)g.YT & 15) == 0));
        if (vec && g.epi == kGemmFwd) epilogue_vec<kGemmFwd>(g, stage, m0, n0, nrows, ncols);
        else if (vec) epilogue_vec<kGemmDx>(g, stage, m0, n0, nrows, ncols);
        else if (g.epi == kGemmFwd) epilogue<kGemmFwd>(g, stage, m0, n0, nrows, ncols);
        else if (g.epi == kGemmDw) epilogue<kGemmDw>(g, stage, m0, n0, nrows, ncols);
        else epilogue<kGemmDx>(g, stage, m0, n0, nrows, ncols);
    }
    // the next kernel may be scheduled while this one tears down (it still waits
    // for this grid's completion before reading what it wrote)
    pdl_trigger();
    if (!ok && tid == 0) set_status(g.status, ROLLOUT_ERR_TIMEOUT);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kBN);
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_group_kernel(const __grid_constant__ GemmGroup grp)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    // which product this block belongs to; each case names its member with a
    // constant index (a dynamic index into the parameter block would make
    // every field access a generic memory load, reloaded after each store)
    int gi = 0;
    while (gi + 1 < grp.n && (int)blockIdx.x >= grp.first[gi + 1]) ++gi;
    const int local = (int)blockIdx.x - grp.first[gi];
    switch (gi) {
    case 0: gemm_cta(grp.g[0], local, sm); break;
    case 1: gemm_cta(grp.g[1], local, sm); break;
    case 2: gemm_cta(grp.g[2], local, sm); break;
    default: gemm_cta(grp.g[3], local, sm); break;
    }
}

}  // namespace

void gemm_plan(GemmArgs &g, int max_split, long long *ws_floats, int *counters)
{
    const int chunks = (g.K + kBK - 1) / kBK;
    const int tiles = ((g.M + kBM - 1) / kBM) * ((g.N + kBN - 1) / kBN);
    int ks = (chunks + 1) / 2;                   // two chunks per split
    if (ks > max_split) ks = max_split;
    if (ks > kMaxSplitG) ks = kMaxSplitG;
    if (ks < 1) ks = 1;
    g.ksplit = ks;
    g.chunks_per_split = (chunks + ks - 1) / ks;
    *ws_floats = ks > 1 ? (long long)tiles * ks * kBM * kBN : 0;
    *counters = ks > 1 ? tiles : 0;
}

cudaError_t launch_gemm_group(const GemmArgs *g, int n, cudaStream_t s)
{
    static std::atomic<unsigned long long> attr{0};   // devices whose attributes are set
    {
        const cudaError_t e_attr = once_per_device(attr, [&]() -> cudaError_t {
            cudaError_t e = cudaFuncSetAttribute(gemm_group_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
            if (e != cudaSuccess) return e;
            return cudaSuccess;
        });
        if (e_attr != cudaSuccess) return e_attr;
    }
    if (n < 1 || n > kGemmGroup) return cudaErrorInvalidValue;
    GemmGroup grp{};
    grp.n = n;
    int blocks = 0;
    for (int i = 0; i < n; ++i) {
        const GemmArgs &a = g[i];
        if (a.M <= 0 || a.N <= 0 || a.K <= 0 || a.ksplit < 1 || a.ksplit > kMaxSplitG ||
            (a.ksplit > 1 && (!a.ws || !a.cnt)))
            return cudaErrorInvalidValue;
        grp.g[i] = a;
        grp.first[i] = blocks;
        blocks += ((a.M + kBM - 1) / kBM) * ((a.N + kBN - 1) / kBN) * a.ksplit;
    }
    grp.first[n] = blocks;
    const cudaError_t e = launch_dependent(gemm_group_kernel, dim3(blocks), dim3(kGemmThreads), kGemmSmem, s, grp);
    return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace rl
