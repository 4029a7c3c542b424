// ppo_gemm.cuh -- the PPO update's tensor-core GEMM (ppo_gemm.cu):
// C[M, N] = A[M, K] B[N, K]^T, float32 in and out, both operands row-major with
// K contiguous, each product taken from a bf16 high/low split of its operands.
#pragma once

#include <cuda_runtime.h>

namespace rl {

enum { kGemmFwd = 0, kGemmDw = 1, kGemmDx = 2 };

struct GemmArgs {
    const float *A = nullptr;   // [M, K], row stride lda (floats)
    int lda = 0;
    const float *B = nullptr;   // [N, K], row stride ldb
    int ldb = 0;
    int M = 0, N = 0, K = 0;
    int epi = kGemmFwd;
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
    int *status = nullptr;      // ROLLOUT_ERR_TIMEOUT if a bounded wait gives up
};

cudaError_t launch_gemm_split(const GemmArgs &g, cudaStream_t s);

}  // namespace rl
