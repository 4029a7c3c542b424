// ppo_gemm.cuh -- the PPO update's tensor-core GEMM (ppo_gemm.cu):
// C[M, N] = A[M, K] B[N, K]^T, float32 in and out, both operands row-major with
// K contiguous, each product taken from a bf16 high/low split of its operands
// (or, for a forward pass in the collector's operand format, from operands
// rounded once to bf16 or tf32).
// Up to kGemmGroup independent products run in one launch; a product may be
// split along K over several CTAs, whose partial tiles the last CTA of each
// tile adds in split order (so the result does not depend on scheduling).
#pragma once

#include <cuda_runtime.h>

namespace rl {

enum { kGemmFwd = 0, kGemmDw = 1, kGemmDx = 2 };
// how the float32 operands enter the tensor cores
enum { kGemmSplit = 0,   // bf16 high + low parts, three MMAs per product (relative error < 1.2e-5)
       kGemmBf16 = 1,    // each operand rounded to bf16 (nearest even), one kind::f16 MMA
       kGemmTf32 = 2,    // each operand rounded to tf32 (nearest, ties away), one kind::tf32 MMA
       kGemmSplit3 = 3 };// bf16 high + middle + low parts, six MMAs per product (relative error < 2^-22)
constexpr int kGemmGroup = 4;
constexpr int kGemmTile = 128;            // C tile: 128 x 128
constexpr int kGemmChunk = 64;            // K elements per chunk

struct GemmArgs {
    const float *A = nullptr;   // [M, K], row stride lda (floats)
    int lda = 0;
    const float *B = nullptr;   // [N, K], row stride ldb
    int ldb = 0;
    int M = 0, N = 0, K = 0;
    int epi = kGemmFwd;
    int operands = kGemmSplit;
    // kGemmFwd: Y = C + bias[n] (ReLU when relu), YT = Y^T (optional)
    const float *bias = nullptr;
    int relu = 0;
    // kGemmDx: Y = C where H[m, n] > 0, else 0; YT = Y^T (optional)
    const float *H = nullptr;
    int ldh = 0;
    float *Y = nullptr;         // [M, N] (row stride ldy); kGemmDw: dW [M, nw]
    int ldy = 0;
    float *YT = nullptr;        // [N, M] (row stride ldt)
    int ldt = 0;
    // kGemmDw: columns n < nw go to Y (dW), column nw to db[m]
    int nw = 0;
    float *db = nullptr;
    // split along K: ksplit CTAs per tile, each taking `chunks_per_split`
    // K-chunks; partial tiles in ws (tiles x ksplit x 128 x 128 floats), one
    // arrival counter per tile in cnt (zero between launches)
    int ksplit = 1, chunks_per_split = 0;
    float *ws = nullptr;
    unsigned int *cnt = nullptr;
    int *status = nullptr;      // ROLLOUT_ERR_TIMEOUT if a bounded wait gives up
};

// fills ksplit / chunks_per_split for a product (at most max_split CTAs per
// tile) and returns the workspace floats and counters it needs
void gemm_plan(GemmArgs &g, int max_split, long long *ws_floats, int *counters);

// launches n (<= kGemmGroup) planned products at once; their ws / cnt regions
// must not overlap
cudaError_t launch_gemm_group(const GemmArgs *g, int n, cudaStream_t s);

}  // namespace rl
