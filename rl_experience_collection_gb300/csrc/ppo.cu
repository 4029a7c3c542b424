// ppo.cu -- the on-device PPO update (include/ppo.h): per mini-batch, the
// actor's log-probabilities are recomputed, the clipped surrogate and the
// critic's squared error are formed and backpropagated, the gradient is
// clipped to a global L2 norm and one Adam step updates actor and critic.
//
// Page "PPO CUDA Pipeline Design -- Zero-Roundtrip Experience Collection",
// the training flow after the collector; page "Fused CUDA Training Kernel --
// Implementation Plan", "Chunk 3: Adam Optimizer Kernel" (norm, clip scale,
// Adam with bias correction and decoupled weight decay).
//
// Parameters, gradients and moments are float32, in the packed weight layout
// (actor, then critic; the curiosity part is carried along untrained).  Each
// dense layer's forward, weight-gradient and input-gradient products are
// float32 GEMMs (cuBLAS, row-major [out, in] weights seen as column-major);
// the gather, bias, ReLU, loss heads, bias gradients, the norm and Adam are the
// kernels below.  Every reduction runs in a fixed order (per column, per
// block, then over the blocks), so a step's result does not depend on timing.
// One optimizer step is captured as a CUDA graph (about 55 launches) and
// replayed for every step of a call: the step's mini-batch slice, statistics
// slot and Adam step count are read from device counters that a last 1-thread
// kernel advances, so that the same graph serves every step.
#include <cublas_v2.h>
#include <math.h>
#include <string.h>

#include <new>

#include "../../include/ppo.h"
#include "internal.cuh"

using namespace rl;

namespace {

constexpr int kMaxLayers = 6;
constexpr int kMaxBatch = 4096;
constexpr int kMaxWidth = 1024;
constexpr int kNormBlocks = 304;   // fixed, so that the norm's summation order is fixed
constexpr int kNormThreads = 256;

constexpr int kGraphMinSteps = 4;              // calls with fewer steps launch directly
constexpr size_t kBlasWorkspace = 32u << 20;   // cuBLAS workspace, fixed so that capture allocates nothing

struct Net {
    int n = 0;
    size_t w[kMaxLayers] = {}, b[kMaxLayers] = {};
    int in[kMaxLayers] = {}, out[kMaxLayers] = {};
};

// what a captured step depends on besides the trainer's own buffers
struct GraphKey {
    const void *ptr[7] = {};           // states, actions, logp_old, adv, ret, indices, stats
    long long T = 0;
    int batch = 0;
    ppo_hparams hp{};
    bool operator==(const GraphKey &o) const
    {
        for (int i = 0; i < 7; ++i)
            if (ptr[i] != o.ptr[i]) return false;
        return T == o.T && batch == o.batch && memcmp(&hp, &o.hp, sizeof hp) == 0;
    }
};

}  // namespace

struct ppo_trainer {
    int device = 0;
    Net net[2];                        // 0 actor, 1 critic
    size_t n_weights = 0, n_trained = 0;
    float *d_w = nullptr, *d_g = nullptr, *d_m = nullptr, *d_v = nullptr;
    long long step = 0;
    // mini-batch buffers, `cap` rows
    int cap = 0;
    float *d_x = nullptr;              // [cap, 54]
    int32_t *d_a = nullptr;
    float *d_lpo = nullptr, *d_adv = nullptr, *d_ret = nullptr;
    float *d_act[2][kMaxLayers] = {};  // layer outputs [cap, out]
    float *d_da = nullptr, *d_db = nullptr;   // backpropagated gradients [cap, kMaxWidth]
    float *d_rows = nullptr;           // per-row statistics [4][cap]
    double *d_part = nullptr;          // [kNormBlocks] partial sums of g^2
    int *d_status = nullptr;
    int *d_k = nullptr;                // step index within the current call
    long long *d_t = nullptr;          // Adam step count
    cublasHandle_t blas = nullptr;
    void *d_ws = nullptr;              // cuBLAS workspace
    cudaStream_t last_stream = nullptr;
    cudaStream_t cap_stream = nullptr; // where one step is captured
    cudaGraphExec_t exec = nullptr;
    GraphKey key;
};

namespace {

int cuda_err(cudaError_t e, const char *what)
{
    return set_error(e == cudaErrorMemoryAllocation ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA, "%s: %s", what,
                     cudaGetErrorString(e));
}

int blas_err(cublasStatus_t st, const char *what)
{
    return set_error(st == CUBLAS_STATUS_ALLOC_FAILED ? ROLLOUT_ERR_NOMEM : ROLLOUT_ERR_CUDA, "%s: cuBLAS status %d",
                     what, (int)st);
}

// ------------------------------------------------------------------ kernels

// one block per mini-batch row: copy the tuple the index names
__global__ void gather_kernel(const float *states, const int32_t *actions, const float *logp_old,
                              const float *adv, const float *ret, long long T, const int32_t *idx_base,
                              const int *step_k, float *x, int32_t *a, float *lpo, float *A, float *R, int *status)
{
    const int r = blockIdx.x;
    long long i = idx_base[(size_t)*step_k * gridDim.x + r];
    if (i < 0 || i >= T) {
        if (threadIdx.x == 0) atomicCAS(status, 0, ROLLOUT_ERR_RANGE);
        i = 0;
    }
    for (int c = threadIdx.x; c < kState; c += blockDim.x) x[(size_t)r * kState + c] = states[i * kState + c];
    if (threadIdx.x == 0) {
        int act = actions[i];
        if (act < 0 || act >= kActions) {
            atomicCAS(status, 0, ROLLOUT_ERR_RANGE);
            act = 0;
        }
        a[r] = act;
        lpo[r] = logp_old[i];
        A[r] = adv[i];
        R[r] = ret[i];
    }
}

// Y[r, j] += b[j], then ReLU for hidden layers
__global__ void bias_act_kernel(float *Y, const float *b, int rows, int n, int relu)
{
    const size_t total = (size_t)rows * n;
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x) {
        const float y = Y[e] + b[e % n];
        Y[e] = (relu && y <= 0.f) ? 0.f : y;
    }
}

// one warp per row: log-softmax of the taken action, ratio, clipped surrogate,
// and the gradient of the loss with respect to the logits
__global__ void actor_head_kernel(const float *logits, const int32_t *a, const float *lpo, const float *A, int B,
                                  float clip_eps, float *dl, float *rows)
{
    const int w = (blockIdx.x * blockDim.x + threadIdx.x) >> 5, lane = threadIdx.x & 31;
    if (w >= B) return;
    const float *l = logits + (size_t)w * kActions;
    const float l0 = l[lane], l1 = lane + 32 < kActions ? l[lane + 32] : -INFINITY;
    float m = fmaxf(l0, l1);
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    const float e0 = expf(l0 - m), e1 = lane + 32 < kActions ? expf(l1 - m) : 0.f;
    float z = e0 + e1;
    for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);
    const int act = a[w];
    const float la = l[act];
    const float logp = (la - m) - logf(z);
    const float rho = expf(logp - lpo[w]);
    const float adv = A[w];
    const float rc = fminf(fmaxf(rho, 1.f - clip_eps), 1.f + clip_eps);
    const float s1 = rho * adv, s2 = rc * adv;
    const bool unclipped = s1 <= s2;
    const float glp = unclipped ? -adv * rho / (float)B : 0.f;
    float *d = dl + (size_t)w * kActions;
    d[lane] = glp * ((lane == act ? 1.f : 0.f) - e0 / z);
    if (lane + 32 < kActions) d[lane + 32] = glp * ((lane + 32 == act ? 1.f : 0.f) - e1 / z);
    if (lane == 0) {
        rows[0 * B + w] = -(unclipped ? s1 : s2);
        rows[2 * B + w] = unclipped ? 0.f : 1.f;
        rows[3 * B + w] = rho;
    }
}

// critic head: squared error and its gradient with respect to v
__global__ void critic_head_kernel(const float *v, const float *R, int B, float value_coef, float *dv, float *rows)
{
    const int r = blockIdx.x * blockDim.x + threadIdx.x;
    if (r >= B) return;
    const float d = v[r] - R[r];
    rows[1 * B + r] = d * d;
    dv[r] = 2.f * value_coef * d / (float)B;
}

// db[j] = sum over rows of dY[r, j] (double): a block takes 32 columns; row
// group y (of 8) sums rows y, y+8, ... in order, then the groups are added in
// order, so the result does not depend on scheduling
constexpr int kBgCols = 32, kBgGroups = 8;
__global__ void __launch_bounds__(kBgCols * kBgGroups) bias_grad_kernel(const float *dY, int rows, int n, float *db)
{
    __shared__ double part[kBgGroups][kBgCols];
    const int c = threadIdx.x % kBgCols, y = threadIdx.x / kBgCols;
    const int j = blockIdx.x * kBgCols + c;
    double s = 0.0;
    if (j < n)
        for (int r = y; r < rows; r += kBgGroups) s += (double)dY[(size_t)r * n + j];
    part[y][c] = s;
    __syncthreads();
    if (y == 0 && j < n) {
        double t = 0.0;
        for (int k = 0; k < kBgGroups; ++k) t += part[k][c];
        db[j] = (float)t;
    }
}

// ReLU' of the layer whose output is H: dX = 0 where H = 0
__global__ void relu_back_kernel(float *dX, const float *H, size_t total)
{
    for (size_t e = blockIdx.x * (size_t)blockDim.x + threadIdx.x; e < total; e += (size_t)gridDim.x * blockDim.x)
        if (!(H[e] > 0.f)) dX[e] = 0.f;
}

__device__ __forceinline__ double block_sum(double v, double *sh)
{
    sh[threadIdx.x] = v;
    __syncthreads();
    for (int s = blockDim.x / 2; s > 0; s >>= 1) {
        if ((int)threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
        __syncthreads();
    }
    const double r = sh[0];
    __syncthreads();
    return r;
}

// partial sums of g^2 over a fixed partition (kNormBlocks blocks)
__global__ void __launch_bounds__(kNormThreads) norm_partial_kernel(const float *g, size_t n, double *part)
{
    __shared__ double sh[kNormThreads];
    double s = 0.0;
    for (size_t i = blockIdx.x * (size_t)kNormThreads + threadIdx.x; i < n; i += (size_t)kNormBlocks * kNormThreads)
        s += (double)g[i] * (double)g[i];
    s = block_sum(s, sh);
    if (threadIdx.x == 0) part[blockIdx.x] = s;
}

// every block first sums the partials in the same order (so all see the same
// norm), then updates its share of the parameters
__global__ void __launch_bounds__(kNormThreads) adam_kernel(float *p, const float *g, float *m, float *v, size_t n,
                                                             const double *part, ppo_hparams hp, const long long *step_t,
                                                             const int *step_k, float *stats)
{
    __shared__ float sh_scale, sh_bc1, sh_bc2;
    if (threadIdx.x == 0) {
        const double t = (double)(*step_t + 1);
        sh_bc1 = (float)(1.0 - pow((double)hp.beta1, t));
        sh_bc2 = (float)(1.0 - pow((double)hp.beta2, t));
        float *norm_out = stats ? stats + (size_t)*step_k * 5 + 4 : nullptr;
        double ss = 0.0;
        for (int b = 0; b < kNormBlocks; ++b) ss += part[b];
        const double norm = sqrt(ss);
        double scale = 1.0;
        if (hp.max_grad_norm > 0.f) scale = fmin(1.0, (double)hp.max_grad_norm / (norm + 1e-6));
        sh_scale = (float)scale;
        if (blockIdx.x == 0 && norm_out) *norm_out = (float)norm;
    }
    __syncthreads();
    const float scale = sh_scale, bc1 = sh_bc1, bc2 = sh_bc2;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const float gi = g[i] * scale;
        const float mi = hp.beta1 * m[i] + (1.f - hp.beta1) * gi;
        const float vi = hp.beta2 * v[i] + (1.f - hp.beta2) * gi * gi;
        m[i] = mi;
        v[i] = vi;
        const float pi = p[i];
        p[i] = pi - (hp.lr * (mi / bc1) / (sqrtf(vi / bc2) + hp.adam_eps) + hp.weight_decay * pi);
    }
}

// means of the four per-row statistics, in row order, into slot step_k of stats
__global__ void stats_kernel(const float *rows, int B, float *stats, const int *step_k)
{
    __shared__ double sh[256];
    float *out = stats + (size_t)*step_k * 5;
    for (int k = 0; k < 4; ++k) {
        double s = 0.0;
        for (int r = threadIdx.x; r < B; r += blockDim.x) s += (double)rows[k * B + r];
        s = block_sum(s, sh);
        if (threadIdx.x == 0) out[k] = (float)(s / B);
    }
}

// the end of a step: the next step's slice and Adam count
__global__ void advance_kernel(int *step_k, long long *step_t)
{
    *step_k += 1;
    *step_t += 1;
}

// ------------------------------------------------------------------ host side

int grid_for(size_t total, int threads)
{
    const size_t b = (total + threads - 1) / threads;
    return (int)(b < 4096 ? b : 4096);
}

void free_batch(ppo_trainer *t)
{
    cudaFree(t->d_x);
    cudaFree(t->d_a);
    cudaFree(t->d_lpo);
    cudaFree(t->d_adv);
    cudaFree(t->d_ret);
    for (auto &net : t->d_act)
        for (float *&p : net) {
            cudaFree(p);
            p = nullptr;
        }
    cudaFree(t->d_da);
    cudaFree(t->d_db);
    cudaFree(t->d_rows);
    t->d_x = nullptr;
    t->d_a = nullptr;
    t->d_lpo = t->d_adv = t->d_ret = t->d_da = t->d_db = t->d_rows = nullptr;
    t->cap = 0;
}

int ensure_batch(ppo_trainer *t, int B)
{
    if (B <= t->cap) return ROLLOUT_OK;
    if (t->exec) {   // the captured step names the old buffers
        cudaGraphExecDestroy(t->exec);
        t->exec = nullptr;
    }
    free_batch(t);   // cudaFree waits for work that may still use the old buffers
    cudaError_t e;
#define ALLOC(p, bytes) if ((e = cudaMalloc(&(p), (bytes))) != cudaSuccess) { free_batch(t); return cuda_err(e, "cudaMalloc(mini-batch)"); }
    ALLOC(t->d_x, (size_t)B * kState * 4);
    ALLOC(t->d_a, (size_t)B * 4);
    ALLOC(t->d_lpo, (size_t)B * 4);
    ALLOC(t->d_adv, (size_t)B * 4);
    ALLOC(t->d_ret, (size_t)B * 4);
    for (int k = 0; k < 2; ++k)
        for (int l = 0; l < t->net[k].n; ++l) ALLOC(t->d_act[k][l], (size_t)B * t->net[k].out[l] * 4);
    ALLOC(t->d_da, (size_t)B * kMaxWidth * 4);
    ALLOC(t->d_db, (size_t)B * kMaxWidth * 4);
    ALLOC(t->d_rows, (size_t)4 * B * 4);
#undef ALLOC
    t->cap = B;
    return ROLLOUT_OK;
}

void free_trainer(ppo_trainer *t)
{
    if (!t) return;
    free_batch(t);
    cudaFree(t->d_w);
    cudaFree(t->d_g);
    cudaFree(t->d_m);
    cudaFree(t->d_v);
    cudaFree(t->d_part);
    cudaFree(t->d_status);
    cudaFree(t->d_k);
    cudaFree(t->d_t);
    if (t->exec) cudaGraphExecDestroy(t->exec);
    if (t->blas) cublasDestroy(t->blas);
    cudaFree(t->d_ws);
    if (t->cap_stream) cudaStreamDestroy(t->cap_stream);
    delete t;
}

const float kOne = 1.f, kZero = 0.f;

// Y[B, out] = X[B, in] W^T (row-major; W is [out, in])
cublasStatus_t gemm_fwd(cublasHandle_t h, const float *W, const float *X, float *Y, int B, int in, int out)
{
    return cublasSgemm(h, CUBLAS_OP_T, CUBLAS_OP_N, out, B, in, &kOne, W, in, X, in, &kZero, Y, out);
}

// dW[out, in] = dY[B, out]^T X[B, in]
cublasStatus_t gemm_dw(cublasHandle_t h, const float *X, const float *dY, float *dW, int B, int in, int out)
{
    return cublasSgemm(h, CUBLAS_OP_N, CUBLAS_OP_T, in, out, B, &kOne, X, in, dY, out, &kZero, dW, in);
}

// dX[B, in] = dY[B, out] W[out, in]
cublasStatus_t gemm_dx(cublasHandle_t h, const float *W, const float *dY, float *dX, int B, int in, int out)
{
    return cublasSgemm(h, CUBLAS_OP_N, CUBLAS_OP_N, in, B, out, &kOne, W, in, dY, out, &kZero, dX, in);
}

// forward of net k over the mini-batch (outputs in d_act[k][*])
int forward(ppo_trainer *t, int k, int B, cudaStream_t s)
{
    const Net &n = t->net[k];
    const float *in = t->d_x;
    for (int l = 0; l < n.n; ++l) {
        cublasStatus_t st = gemm_fwd(t->blas, t->d_w + n.w[l], in, t->d_act[k][l], B, n.in[l], n.out[l]);
        if (st != CUBLAS_STATUS_SUCCESS) return blas_err(st, "forward GEMM");
        const size_t total = (size_t)B * n.out[l];
        bias_act_kernel<<<grid_for(total, 256), 256, 0, s>>>(t->d_act[k][l], t->d_w + n.b[l], B, n.out[l],
                                                             l < n.n - 1);
        in = t->d_act[k][l];
    }
    return ROLLOUT_OK;
}

// backward of net k from the gradient at its output (in d_da), into d_g
int backward(ppo_trainer *t, int k, int B, cudaStream_t s)
{
    const Net &n = t->net[k];
    float *dy = t->d_da, *dx = t->d_db;
    for (int l = n.n - 1; l >= 0; --l) {
        const float *in = l == 0 ? t->d_x : t->d_act[k][l - 1];
        cublasStatus_t st = gemm_dw(t->blas, in, dy, t->d_g + n.w[l], B, n.in[l], n.out[l]);
        if (st != CUBLAS_STATUS_SUCCESS) return blas_err(st, "weight-gradient GEMM");
        bias_grad_kernel<<<(n.out[l] + kBgCols - 1) / kBgCols, kBgCols * kBgGroups, 0, s>>>(dy, B, n.out[l],
                                                                                          t->d_g + n.b[l]);
        if (l == 0) break;
        st = gemm_dx(t->blas, t->d_w + n.w[l], dy, dx, B, n.in[l], n.out[l]);
        if (st != CUBLAS_STATUS_SUCCESS) return blas_err(st, "input-gradient GEMM");
        const size_t total = (size_t)B * n.in[l];
        relu_back_kernel<<<grid_for(total, 256), 256, 0, s>>>(dx, t->d_act[k][l - 1], total);
        float *tmp = dy;
        dy = dx;
        dx = tmp;
    }
    return ROLLOUT_OK;
}

int check_update_args(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                      const float *adv, const float *ret, long long T, const int32_t *indices, int batch,
                      const ppo_hparams *hp)
{
    if (!t || !hp) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    if (!states || !actions || !logp_old || !adv || !ret || !indices)
        return set_error(ROLLOUT_ERR_INVALID, "null array argument");
    if (T < 1 || T > (1LL << 31) - 1) return set_error(ROLLOUT_ERR_INVALID, "T must be in [1, 2^31)");
    if (batch < 1 || batch > kMaxBatch) return set_error(ROLLOUT_ERR_INVALID, "batch must be in [1, %d]", kMaxBatch);
    const float hv[] = {hp->clip_eps, hp->value_coef, hp->lr, hp->beta1, hp->beta2, hp->adam_eps, hp->max_grad_norm,
                        hp->weight_decay};
    for (float f : hv)
        if (!isfinite(f)) return set_error(ROLLOUT_ERR_INVALID, "hyperparameters must be finite");
    if (hp->clip_eps < 0.f || hp->lr < 0.f || hp->adam_eps <= 0.f || !(hp->beta1 >= 0.f && hp->beta1 < 1.f) ||
        !(hp->beta2 >= 0.f && hp->beta2 < 1.f))
        return set_error(ROLLOUT_ERR_INVALID, "need clip_eps >= 0, lr >= 0, adam_eps > 0, beta1 and beta2 in [0, 1)");
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_err(e, "cudaGetDevice");
    if (dev != t->device) return set_error(ROLLOUT_ERR_INVALID, "current device is not the trainer's");
    return ensure_batch(t, batch);
}

// the loss statistics (per row, in d_rows) and the gradient (d_g) of the
// mini-batch rows[d_k * B .. d_k * B + B) at the current weights
int loss_gradient(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                  const float *adv, const float *ret, long long T, const int32_t *rows, int B, const ppo_hparams *hp,
                  cudaStream_t s)
{
    int rc;
    gather_kernel<<<B, 64, 0, s>>>(states, actions, logp_old, adv, ret, T, rows, t->d_k, t->d_x, t->d_a, t->d_lpo,
                                   t->d_adv, t->d_ret, t->d_status);
    // actor: log-probs, surrogate, its gradient
    if ((rc = forward(t, 0, B, s))) return rc;
    actor_head_kernel<<<(B * 32 + 255) / 256, 256, 0, s>>>(t->d_act[0][2], t->d_a, t->d_lpo, t->d_adv, B,
                                                           hp->clip_eps, t->d_da, t->d_rows);
    if ((rc = backward(t, 0, B, s))) return rc;
    // critic: squared error, its gradient
    if ((rc = forward(t, 1, B, s))) return rc;
    critic_head_kernel<<<(B + 255) / 256, 256, 0, s>>>(t->d_act[1][kCriticLayers - 1], t->d_ret, B, hp->value_coef,
                                                       t->d_da, t->d_rows);
    return backward(t, 1, B, s);
}

// one optimizer step (the counters pick the mini-batch, the statistics slot and t)
int step(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old, const float *adv,
         const float *ret, long long T, const int32_t *indices, int B, const ppo_hparams *hp, float *stats,
         cudaStream_t s)
{
    cublasStatus_t st = cublasSetStream(t->blas, s);
    if (st != CUBLAS_STATUS_SUCCESS) return blas_err(st, "cublasSetStream");
    int rc = loss_gradient(t, states, actions, logp_old, adv, ret, T, indices, B, hp, s);
    if (rc) return rc;
    norm_partial_kernel<<<kNormBlocks, kNormThreads, 0, s>>>(t->d_g, t->n_trained, t->d_part);
    adam_kernel<<<kNormBlocks, kNormThreads, 0, s>>>(t->d_w, t->d_g, t->d_m, t->d_v, t->n_trained, t->d_part, *hp,
                                                     t->d_t, t->d_k, stats);
    if (stats) stats_kernel<<<1, 256, 0, s>>>(t->d_rows, B, stats, t->d_k);
    advance_kernel<<<1, 1, 0, s>>>(t->d_k, t->d_t);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "PPO step launch");
}

// the graph of one step for these arguments (captured on the trainer's own
// stream; reused while the arguments stay the same)
int step_graph(ppo_trainer *t, const GraphKey &key, const float *states, const int32_t *actions,
               const float *logp_old, const float *adv, const float *ret, long long T, const int32_t *indices, int B,
               const ppo_hparams *hp, float *stats)
{
    if (t->exec && t->key == key) return ROLLOUT_OK;
    if (t->exec) {
        cudaGraphExecDestroy(t->exec);
        t->exec = nullptr;
    }
    cudaError_t e = cudaStreamBeginCapture(t->cap_stream, cudaStreamCaptureModeThreadLocal);
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamBeginCapture");
    int rc = step(t, states, actions, logp_old, adv, ret, T, indices, B, hp, stats, t->cap_stream);
    cudaGraph_t g = nullptr;
    e = cudaStreamEndCapture(t->cap_stream, &g);
    if (rc) {
        if (g) cudaGraphDestroy(g);
        return rc;
    }
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamEndCapture");
    e = cudaGraphInstantiate(&t->exec, g, 0);
    cudaGraphDestroy(g);
    if (e != cudaSuccess) {
        t->exec = nullptr;
        return cuda_err(e, "cudaGraphInstantiate");
    }
    t->key = key;
    return ROLLOUT_OK;
}

}  // namespace

extern "C" {

int ppo_create(const float *weights, const rollout_dims *dims, ppo_trainer **out)
{
    clear_error();
    if (!weights || !dims || !out) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    int rc = validate_dims(dims);
    if (rc) return rc;
    ppo_trainer *t = new (std::nothrow) ppo_trainer();
    if (!t) return set_error(ROLLOUT_ERR_NOMEM, "host allocation failed");
    // packed layout: actor (3 layers), critic (5 hidden + head), curiosity (2 layers)
    size_t off = 0;
    const int ain[3] = {kState, kActorH1, kActorH2}, aout[3] = {kActorH1, kActorH2, kActions};
    Net &A = t->net[0], &Cn = t->net[1];
    A.n = 3;
    for (int l = 0; l < 3; ++l) {
        A.in[l] = ain[l];
        A.out[l] = aout[l];
        A.w[l] = off; off += (size_t)ain[l] * aout[l];
        A.b[l] = off; off += aout[l];
    }
    Cn.n = kCriticLayers;
    int prev = kState;
    for (int l = 0; l < kCriticLayers; ++l) {
        const int o = l < 5 ? dims->critic_h[l] : 1;
        Cn.in[l] = prev;
        Cn.out[l] = o;
        Cn.w[l] = off; off += (size_t)prev * o;
        Cn.b[l] = off; off += o;
        prev = o;
    }
    t->n_trained = off;
    off += (size_t)(kState + kActions) * kCurH + kCurH + (size_t)kCurH * kState + kState;
    t->n_weights = off;
    cudaError_t e = cudaGetDevice(&t->device);
    if (e != cudaSuccess) { free_trainer(t); return cuda_err(e, "cudaGetDevice"); }
    if ((e = cudaMalloc(&t->d_w, t->n_weights * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_g, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_m, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_v, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMalloc(&t->d_part, kNormBlocks * sizeof(double))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_status, sizeof(int))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_k, sizeof(int))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_t, sizeof(long long))) != cudaSuccess ||
        (e = cudaMalloc(&t->d_ws, kBlasWorkspace)) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "cudaMalloc(trainer)");
    }
    if ((e = cudaStreamCreateWithFlags(&t->cap_stream, cudaStreamNonBlocking)) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "cudaStreamCreateWithFlags");
    }
    if ((e = cudaMemcpy(t->d_w, weights, t->n_weights * 4, cudaMemcpyHostToDevice)) != cudaSuccess ||
        (e = cudaMemset(t->d_m, 0, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMemset(t->d_v, 0, t->n_trained * 4)) != cudaSuccess ||
        (e = cudaMemset(t->d_status, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(t->d_k, 0, sizeof(int))) != cudaSuccess ||
        (e = cudaMemset(t->d_t, 0, sizeof(long long))) != cudaSuccess) {
        free_trainer(t);
        return cuda_err(e, "trainer upload");
    }
    cublasStatus_t st = cublasCreate(&t->blas);
    if (st != CUBLAS_STATUS_SUCCESS) { free_trainer(t); return blas_err(st, "cublasCreate"); }
    // float32 GEMMs: no TF32 or other reduced-precision math
    if ((st = cublasSetMathMode(t->blas, CUBLAS_PEDANTIC_MATH)) != CUBLAS_STATUS_SUCCESS ||
        (st = cublasSetWorkspace(t->blas, t->d_ws, kBlasWorkspace)) != CUBLAS_STATUS_SUCCESS) {
        free_trainer(t);
        return blas_err(st, "cuBLAS setup");
    }
    *out = t;
    return ROLLOUT_OK;
}

int ppo_update(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
               const float *adv, const float *ret, long long T, const int32_t *indices, int n_steps, int batch,
               const ppo_hparams *hp, float *stats, void *stream)
{
    clear_error();
    if (n_steps < 0) return set_error(ROLLOUT_ERR_INVALID, "n_steps must be >= 0");
    int rc = check_update_args(t, states, actions, logp_old, adv, ret, T, indices, batch, hp);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    t->last_stream = s;
    if (n_steps == 0) return ROLLOUT_OK;
    cudaError_t e = cudaMemsetAsync(t->d_k, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_err(e, "cudaMemsetAsync(step index)");
    if (n_steps >= kGraphMinSteps) {
        GraphKey key;
        const void *ptrs[7] = {states, actions, logp_old, adv, ret, indices, stats};
        memcpy(key.ptr, ptrs, sizeof ptrs);
        key.T = T;
        key.batch = batch;
        key.hp = *hp;
        if ((rc = step_graph(t, key, states, actions, logp_old, adv, ret, T, indices, batch, hp, stats))) return rc;
        for (int k = 0; k < n_steps; ++k)
            if ((e = cudaGraphLaunch(t->exec, s)) != cudaSuccess) return cuda_err(e, "cudaGraphLaunch");
    } else {
        for (int k = 0; k < n_steps; ++k)
            if ((rc = step(t, states, actions, logp_old, adv, ret, T, indices, batch, hp, stats, s))) return rc;
    }
    t->step += n_steps;
    return ROLLOUT_OK;
}

int ppo_gradient(ppo_trainer *t, const float *states, const int32_t *actions, const float *logp_old,
                 const float *adv, const float *ret, long long T, const int32_t *indices, int batch,
                 const ppo_hparams *hp, float *grad, float *stats, void *stream)
{
    clear_error();
    if (!grad) return set_error(ROLLOUT_ERR_INVALID, "null gradient buffer");
    int rc = check_update_args(t, states, actions, logp_old, adv, ret, T, indices, batch, hp);
    if (rc) return rc;
    cudaStream_t s = (cudaStream_t)stream;
    t->last_stream = s;
    cublasStatus_t st = cublasSetStream(t->blas, s);
    if (st != CUBLAS_STATUS_SUCCESS) return blas_err(st, "cublasSetStream");
    cudaError_t e = cudaMemsetAsync(t->d_k, 0, sizeof(int), s);
    if (e != cudaSuccess) return cuda_err(e, "cudaMemsetAsync(step index)");
    if ((rc = loss_gradient(t, states, actions, logp_old, adv, ret, T, indices, batch, hp, s))) return rc;
    if (stats) stats_kernel<<<1, 256, 0, s>>>(t->d_rows, batch, stats, t->d_k);
    e = cudaMemcpyAsync(grad, t->d_g, t->n_trained * 4, cudaMemcpyDefault, s);
    if (e == cudaSuccess) e = cudaGetLastError();
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "PPO gradient");
}

int ppo_get_weights(ppo_trainer *t, float *weights, void *stream)
{
    clear_error();
    if (!t || !weights) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    cudaError_t e = cudaMemcpyAsync(weights, t->d_w, t->n_weights * 4, cudaMemcpyDefault, (cudaStream_t)stream);
    return e == cudaSuccess ? ROLLOUT_OK : cuda_err(e, "cudaMemcpyAsync(weights)");
}

int ppo_device_weights(ppo_trainer *t, const float **weights)
{
    clear_error();
    if (!t || !weights) return set_error(ROLLOUT_ERR_INVALID, "null argument");
    *weights = t->d_w;
    return ROLLOUT_OK;
}

int ppo_reset_optimizer(ppo_trainer *t, void *stream)
{
    clear_error();
    if (!t) return set_error(ROLLOUT_ERR_INVALID, "null trainer");
    cudaError_t e;
    if ((e = cudaMemsetAsync(t->d_m, 0, t->n_trained * 4, (cudaStream_t)stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(t->d_v, 0, t->n_trained * 4, (cudaStream_t)stream)) != cudaSuccess ||
        (e = cudaMemsetAsync(t->d_t, 0, sizeof(long long), (cudaStream_t)stream)) != cudaSuccess)
        return cuda_err(e, "cudaMemsetAsync(moments)");
    t->step = 0;
    return ROLLOUT_OK;
}

int ppo_status(ppo_trainer *t)
{
    clear_error();
    if (!t) return set_error(ROLLOUT_ERR_INVALID, "null trainer");
    cudaError_t e = cudaStreamSynchronize(t->last_stream);
    if (e != cudaSuccess) return cuda_err(e, "cudaStreamSynchronize");
    int st = 0;
    if ((e = cudaMemcpy(&st, t->d_status, sizeof(int), cudaMemcpyDeviceToHost)) != cudaSuccess ||
        (e = cudaMemset(t->d_status, 0, sizeof(int))) != cudaSuccess)
        return cuda_err(e, "status read");
    return st;
}

void ppo_destroy(ppo_trainer *t)
{
    if (!t) return;
    cudaDeviceSynchronize();
    free_trainer(t);
}

}  // extern "C"
