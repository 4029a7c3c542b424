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
// One CTA computes a 128 x 128 tile of C: its 128 threads load the tile's
// K-chunks of A and B (64 elements each, zero outside the matrices), split
// them into swizzled bf16 operand tiles in shared memory (two stages, so that
// loading chunk c + 1 overlaps the MMAs of chunk c), one thread issues the
// MMAs, and after the last chunk each thread takes one row of the accumulator
// from tensor memory through the epilogue:
//   forward:         Y = C + bias (ReLU for hidden layers), and Y^T
//   weight gradient: C[:, :nw] into dW, column nw into db (the B operand's
//                    row nw is all ones: the column sums of dY)
//   input gradient:  Y = C where H > 0, else 0 (ReLU'), and Y^T
// Every wait is bounded; a CTA that gives up sets ROLLOUT_ERR_TIMEOUT.
#include "env.cuh"
#include "ppo_gemm.cuh"
#include "umma.cuh"

namespace rl {

namespace {

using namespace umma;

constexpr int kBM = 128, kBN = 128, kBK = 64;            // tile rows, columns, K elements per chunk
constexpr int kTile = 128 * 128;                           // bytes of one 128-row bf16 operand tile
constexpr int kStageBytes = 4 * kTile;                     // A hi, A lo, B hi, B lo
constexpr int kGemmSmem = 2 * kStageBytes + 1024;          // two stages + alignment slack
constexpr int kGemmThreads = 128;

// the bf16 pair (hi, lo) of x
__device__ __forceinline__ void split_bf16(float x, float &hi, float &lo)
{
    const uint32_t h = pack_bf16x2(0.f, x) & 0xFFFF0000u;   // nearest-even bf16 of x (upper half)
    hi = __uint_as_float(h);
    lo = x - hi;                                             // exact in float32
}

// loads K-chunk c of rows [r0, r0 + 128) of X [rows, K] (row stride ld) into
// the swizzled hi / lo tiles; thread t takes 16 runs of four elements
__device__ __forceinline__ void load_split(const float *X, int ld, int rows, int K, int r0, int c, uint8_t *hi_tile,
                                           uint8_t *lo_tile)
{
    const int tid = threadIdx.x;
#pragma unroll 4
    for (int s = 0; s < (kBM * kBK / 4) / kGemmThreads; ++s) {
        const int j = tid + kGemmThreads * s;                   // run of four elements
        const int r = j >> 4, q = j & 15;                        // row, run within the row
        const int row = r0 + r, col = c * kBK + 4 * q;
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = (row < rows && col + i < K) ? __ldg(X + (long long)row * ld + col + i) : 0.f;
        float h[4], l[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) split_bf16(v[i], h[i], l[i]);
        const uint2 ph = make_uint2(pack_bf16x2(h[0], h[1]), pack_bf16x2(h[2], h[3]));
        const uint2 pl = make_uint2(pack_bf16x2(l[0], l[1]), pack_bf16x2(l[2], l[3]));
        const uint32_t off = sw128_offset(r, q >> 1) + 8 * (q & 1);   // 16-byte unit q/2 of row r, half q%2
        *reinterpret_cast<uint2 *>(hi_tile + off) = ph;
        *reinterpret_cast<uint2 *>(lo_tile + off) = pl;
    }
}

__global__ void __launch_bounds__(kGemmThreads, 1) gemm_split_kernel(GemmArgs g)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    __shared__ __align__(8) uint64_t bar_done[2], bar_final;
    __shared__ uint32_t tmem_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int m0 = blockIdx.x * kBM, n0 = blockIdx.y * kBN;
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
    const uint32_t tmem = tmem_sh;
    volatile int *abort = &abort_sh;
    const int chunks = (g.K + kBK - 1) / kBK;
    constexpr uint32_t id = idesc(true, kBM, kBN);
    bool ok = true;
    for (int c = 0; c < chunks; ++c) {
        const int s = c & 1;
        uint8_t *st = sm + s * kStageBytes;
        // the MMAs of chunk c - 2 read this stage: wait until they are done
        if (c >= 2) ok = __syncthreads_and(ok && mbar_wait(&bar_done[s], (uint32_t)(((c - 2) >> 1) & 1), abort));
        if (!ok) break;
        load_split(g.A, g.lda, g.M, g.K, m0, c, st, st + kTile);
        load_split(g.B, g.ldb, g.N, g.K, n0, c, st + 2 * kTile, st + 3 * kTile);
        fence_async_smem();                       // generic-proxy stores -> visible to the tensor core
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const uint32_t a_hi = smem_u32(st), a_lo = a_hi + kTile, b_hi = a_hi + 2 * kTile, b_lo = a_hi + 3 * kTile;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t acc = (c > 0 || k > 0) ? 1u : 0u;
                mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_hi + 32 * k), id, acc);
                mma<true>(tmem, desc_sw128(a_hi + 32 * k), desc_sw128(b_lo + 32 * k), id, 1u);
                mma<true>(tmem, desc_sw128(a_lo + 32 * k), desc_sw128(b_hi + 32 * k), id, 1u);
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
    if (ok && chunks > 0) {
        const int r = tid, m = m0 + r;
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
        for (int cb = 0; cb < kBN; cb += 32) {
            if (n0 + cb >= g.N) break;                             // CTA-uniform
            float v[32];
            tmem_ld32(lane_addr + cb, v);
            tmem_ld_wait();
            if (m >= g.M) continue;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int n = n0 + cb + i;
                if (n >= g.N) continue;
                float y = v[i];
                if (g.epi == kGemmFwd) {
                    y += __ldg(g.bias + n);
                    if (g.relu) y = relu(y);
                } else if (g.epi == kGemmDx) {
                    y = __ldg(g.H + (long long)m * g.ldh + n) > 0.f ? y : 0.f;
                }
                if (g.epi == kGemmDw) {
                    if (n < g.nw) g.Y[(long long)m * g.ldy + n] = y;
                    else g.db[m] = y;
                } else {
                    g.Y[(long long)m * g.ldy + n] = y;
                    if (g.YT) g.YT[(long long)n * g.ldt + m] = y;
                }
            }
        }
    } else if (!ok && tid == 0) {
        set_status(g.status, ROLLOUT_ERR_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kBN);
}

}  // namespace

cudaError_t launch_gemm_split(const GemmArgs &g, cudaStream_t s)
{
    static bool attr = false;
    if (!attr) {
        cudaError_t e = cudaFuncSetAttribute(gemm_split_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (g.M <= 0 || g.N <= 0 || g.K <= 0) return cudaErrorInvalidValue;
    const dim3 grid((g.M + kBM - 1) / kBM, (g.N + kBN - 1) / kBN);
    gemm_split_kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(g);
    return cudaGetLastError();
}

}  // namespace rl
